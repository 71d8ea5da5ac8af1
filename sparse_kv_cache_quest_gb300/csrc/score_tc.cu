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
// all segments form one range, split evenly over a persistent grid of two CTAs
// per SM (two MMA lanes and rings side by side: a lane blocks while its MMAs
// run, and each CTA holds one query-operand buffer, rebuilt when its segment
// changes).  A tile is moved as its kmax chunks, then its kmin chunks, through
// a ring of stages that each hold one piece of a half: the whole half, or,
// where only two half-sized stages fit beside the query operand, half of it
// (16 KiB at d_h 128), so that a stage is held only while the few MMAs that
// read it run (pieces()).  Roles in a CTA (warp-specialised, mbarrier
// hand-offs, every wait bounded):
//   warp 0, one lane  - one 3-D TMA tensor copy per piece (a box of CH /
//                       pieces chunks x 128 blocks x 8 dims of the chunk-major
//                       summaries; 16-byte bulk copies per chunk when the block
//                       count is not a multiple of 8);
//   warp 1, one lane  - the piece's MMAs (K = 16 each) into one of four TMEM
//                       accumulators (the warp also owns the TMEM allocation);
//   warps 2-5 (scan)  - per segment, the split query operand {q+, q-} in the
//                       no-swizzle K-major layout, Q_d and max_d Q_d (built
//                       once the previous segment's MMAs are done); without wrong-side
//                       sums also, per piece, C_b's share from the stage
//                       (each thread one block row), after which the stage is
//                       released, and C_b to the TMEM warps through a small ring;
//   warps 6-9 (TMEM)  - the accumulator row (tcgen05.ld), the max over the
//                       columns, the radius (with wrong-side sums, C_b = max_d
//                       Q_d * wsum_b from a load issued a tile ahead), the stores.
// The scan warps move with the copies and the TMEM warps with the MMAs, so
// neither holds up the other's ring; the tile walk and the ring positions are
// kept as counters (a 64-bit division on the single MMA lane costs more than
// the MMAs it issues).
// Shared-memory operands use the no-swizzle K-major layout of 8-row x 16-byte
// core matrices: the chunk-major summaries already are that layout (chunk c of
// 128 blocks = 16 core matrices at 128-byte steps), so a piece lands as is:
// LBO (next 8 K-elements) = 2048 bytes, SBO (next 8 rows) = 128.
#include <algorithm>
#include <cfloat>

#include "common.cuh"

namespace oasis {
namespace {

constexpr int kRows = 128;                    // blocks per tile (MMA M)
constexpr int kGroupWarps = 4;                // scan warps, and TMEM warps
constexpr int kThreadsTC = 32 * (2 + 2 * kGroupWarps);
constexpr int kNAcc = 4;                      // TMEM accumulators
constexpr int kNC = 4;                        // C_b hand-off ring (scan -> TMEM warps)
constexpr uint32_t kChunkBytes = kRows * 16;  // one 8-dim chunk of a tile
constexpr uint32_t kWaitTriesTC = 1u << 22;   // bounded mbarrier polls (far beyond any real copy or MMA)
constexpr int kCtasPerSm = 2;                 // CTAs per SM: two MMA lanes and rings side by side
constexpr int kMaxRegsTC = 80;                // registers a thread (see the kernel)
constexpr int kBBufs = 1;                     // query-operand buffers per CTA
constexpr size_t kSmemCap = (228 * 1024) / kCtasPerSm - 1024;  // per CTA (1 KiB of each SM's share is reserved)
constexpr int kMaxStages = 16;

// Shared memory of a CTA besides its ring: the query operand, Q (two slots),
// the C_b ring, max_d Q_d (two slots), the barriers and the TMEM address.
template <int N, int CH>
constexpr size_t fixed_smem() {
  return kBBufs * static_cast<size_t>(N) * 2 * (CH * 8) * 2 + (2 * CH * 8 + kNC * kRows + 2) * sizeof(float) +
         (2 * kMaxStages + 2 * kNAcc + 8 + 2 * kNC + 1) * sizeof(uint64_t) + 16;
}
// Ring stages (pieces) per half-tile.  Where only two half-tile stages fit
// beside the query operand (32 to 64 query columns at d_h 128), a stage spends
// a large share of its turn held under its MMAs; halves cut in two keep more of
// the same ring in flight (235B-shaped layer, 64 columns: 47.8 -> 47.4 us).  With
// three or more half-tile stages the extra copies and barrier rounds cost more
// than that gains (Qwen3-8B-shaped step, 16 columns: 45.3-45.9 -> 47.1 us), so
// the halves stay whole.
template <int N, int CH>
constexpr int pieces() {
  return (kSmemCap - fixed_smem<N, CH>()) / (static_cast<size_t>(CH) * kChunkBytes) >= 3 ? 1 : 2;
}

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
__device__ __forceinline__ void scan_barrier() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kGroupWarps) : "memory"); }
// one 3-D tensor copy (x, y, z) into this CTA's shared memory, completing on bar;
// the summaries are read once per step, so their L2 lines are marked evict-first
// (as the attention's slot tiles: data other kernels of the step reuse stays in
// L2; this kernel alone 47.6 -> 46.8 us on the 235B-shaped layer)
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, %4}], "
      "[%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

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

// The CTA's tiles [t0, t1) in segment-major order (tile j of segment s =
// blocks j*kRows .. of s, global index t = s*tps + j); a tile is work when its
// first block is a candidate of its segment.  begin() divides once; advance()
// steps without dividing and reads a segment's length when it enters it.
struct TileIter {
  int64_t t0, t1;
  int tps, Hkv, W, Nb_max;
  const int32_t *seq_len;
  int s = 0, j = 0, nc = 0;  // the current work tile: segment, tile in it, candidates of the segment
  int64_t t = 0;
  __device__ int nc_of(int seg) const {
    int L = __ldg(seq_len + seg / Hkv);
    L = L < 0 ? 0 : (L > Nb_max * kBlockTokens ? Nb_max * kBlockTokens : L);
    return ceil_div(L, kBlockTokens) - W;
  }
  // the first work tile at or after the current position (t = t1 if none)
  __device__ void settle() {
    while (t < t1) {
      if (j < tps && j * kRows < nc) return;
      ++s;
      j = 0;
      t = static_cast<int64_t>(s) * tps;
      if (t >= t1) {
        t = t1;
        return;
      }
      nc = nc_of(s);
    }
  }
  __device__ void begin() {
    s = static_cast<int>(t0 / tps);
    j = static_cast<int>(t0 - static_cast<int64_t>(s) * tps);
    t = t0;
    nc = t0 < t1 ? nc_of(s) : 0;
    settle();
  }
  __device__ bool valid() const { return t < t1; }
  __device__ void advance() {
    ++j;
    ++t;
    settle();
  }
  // does segment seg have a work tile in [t0, t1)?
  __device__ bool active(int seg) const {
    const int64_t first = std::max<int64_t>(t0, static_cast<int64_t>(seg) * tps);
    return static_cast<int>(first - static_cast<int64_t>(seg) * tps) * kRows < nc_of(seg);
  }
};

template <int N, int CH>
// 80 registers a thread (no spills): two CTAs then take 51,200 of an SM's
// 65,536, which leaves room on the same SM for a selection or a staging CTA of
// another layer (at 96 they took 61,440 and any such CTA cost the SM one of its
// scoring CTAs, started a wave late)
__global__ void __maxnreg__(kMaxRegsTC)
    k_score_tc(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmn, bool use_tma,
               const uint16_t *__restrict__ kmin, const uint16_t *__restrict__ kmax,
               const float *__restrict__ wsum, int Nb_max, const uint16_t *__restrict__ qdraft, int S, int Hkv,
               int G, int Nd, const int32_t *__restrict__ seq_len, int W, float *__restrict__ scores,
               float *__restrict__ radius, int32_t *status, int tps, int stages) {
  constexpr int D = CH * 8;
  constexpr int kPieces = pieces<N, CH>();
  constexpr int CP = CH / kPieces;                     // chunks per piece (a ring stage)
  constexpr int KP = CP / 2;                           // MMAs per piece (K = 16 each)
  constexpr uint32_t kPiece = CP * kChunkBytes;        // a piece: CP chunks of the kmax or the kmin half-tile
  static_assert(CH % kPieces == 0 && CP % 2 == 0, "a piece holds whole MMA K-steps");
  constexpr uint32_t kBBytes = static_cast<uint32_t>(N) * 2 * D * 2;
  constexpr uint32_t kTmemCols = kNAcc * N <= 64 ? 64 : (kNAcc * N <= 128 ? 128 : 256);
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *sA = smem;                                               // [stages][kPiece]
  uint8_t *sB = sA + static_cast<size_t>(stages) * kPiece;          // [kBBufs][kBBytes]
  float *sQ = reinterpret_cast<float *>(sB + kBBufs * kBBytes);     // [2][D]
  float *sC = sQ + 2 * D;                                           // [kNC][kRows]
  float *sQmax = sC + kNC * kRows;                                  // [2]: max_d Q_d per query buffer
  uint64_t *bars = reinterpret_cast<uint64_t *>(sQmax + 2);
  uint64_t *full = bars, *empty = full + stages, *accF = empty + stages, *accE = accF + kNAcc;
  uint64_t *bqF = accE + kNAcc, *bqE = bqF + 2, *qmF = bqE + 2, *qmE = qmF + 2, *cF = qmE + 2, *cE = cF + kNC;
  uint64_t *drain = cE + kNC;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
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
      // the MMAs' commit, plus each scan warp when it reads the stage (no wsum)
      mbar_init(&empty[i], wsum != nullptr ? 1 : 1 + kGroupWarps);
    }
    for (int i = 0; i < kNAcc; ++i) {
      mbar_init(&accF[i], 1);
      mbar_init(&accE[i], kGroupWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bqF[i], 32 * kGroupWarps);
      mbar_init(&bqE[i], 1);
      mbar_init(&qmF[i], 1);            // max_d Q_d of the buffer's segment is in sQmax
      mbar_init(&qmE[i], kGroupWarps);  // every TMEM warp has taken it
    }
    for (int i = 0; i < kNC; ++i) {
      mbar_init(&cF[i], 32 * kGroupWarps);
      mbar_init(&cE[i], kGroupWarps);
    }
    mbar_init(drain, 1);
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
    // ---------------- producer: one copy per piece into the stage ring
    if (lane == 0) {
      int64_t issued = 0;    // pieces
      int st = 0;            // issued % stages
      uint32_t round = 0;    // issued / stages
      bool ok = true;
      for (it.begin(); it.valid() && ok; it.advance()) {
        const int s = it.s;
        const int base = it.j * kRows;
        const int rows = min(kRows, it.nc - base);
#pragma unroll 1
        for (int q = 0; q < 2 * kPieces; ++q) {  // the kmax pieces, then the kmin pieces
          const int h = q / kPieces, c0 = (q % kPieces) * CP;
          if (issued >= stages && !wait_or_abort(&empty[st], (round - 1u) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t *dst = sA + static_cast<size_t>(st) * kPiece;
          if (use_tma) {
            // box {8 blocks x 8 dims, 16 groups of 8 blocks, CP chunks}: rows past
            // the summary capacity arrive zero-filled, so the byte count is fixed
            mbar_arrive_expect_tx(&full[st], kPiece);
            tma_load_3d(dst, h == 0 ? &tmx : &tmn, 0, base / 8, s * CH + c0, &full[st]);
          } else {
            const uint32_t bytes = static_cast<uint32_t>(rows) * 16u;
            mbar_arrive_expect_tx(&full[st], CP * bytes);
            const uint4 *g = reinterpret_cast<const uint4 *>(h == 0 ? kmax : kmin) +
                             static_cast<int64_t>(s * CH + c0) * Nb_max + base;
#pragma unroll 4
            for (int c = 0; c < CP; ++c)
              bulk_g2s(dst + c * kChunkBytes, g + static_cast<int64_t>(c) * Nb_max, bytes, &full[st]);
          }
          ++issued;
          if (++st == stages) {
            st = 0;
            ++round;
          }
        }
      }
      // never leave with copies in flight: wait for the last stages issued
      for (int64_t k = std::max<int64_t>(0, issued - stages); k < issued; ++k)
        mbar_wait_bounded(&full[k % stages], static_cast<uint32_t>(k / stages) & 1u, kWaitTriesTC);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16<N>();
      int64_t i = 0, u = 0;  // tiles, pieces
      int st = 0;            // u % stages
      uint32_t round = 0;    // u / stages
      int seg_prev = -1, nseg = 0, buf = 0;
      bool ok = true;
      for (it.begin(); it.valid() && ok; it.advance()) {
        const int s = it.s;
        if (s != seg_prev) {  // the query operand of this segment
          if (seg_prev >= 0) tc_commit(&bqE[buf]);  // the previous segment's operand is free once its MMAs are done
          buf = nseg % kBBufs;
          ok = wait_or_abort(&bqF[buf], static_cast<uint32_t>(nseg / kBBufs) & 1u, abort_flag);
          ++nseg;
          seg_prev = s;
          if (!ok) break;
        }
        const int acc = static_cast<int>(i % kNAcc);
        if (i >= kNAcc &&
            !wait_or_abort(&accE[acc], static_cast<uint32_t>((i / kNAcc) - 1) & 1u, abort_flag))
          break;
        const uint32_t b0 = smem_addr(sB + static_cast<size_t>(buf) * kBBytes);
#pragma unroll 1
        for (int q = 0; q < 2 * kPieces && ok; ++q) {
          ok = wait_or_abort(&full[st], round & 1u, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a0 = smem_addr(sA + static_cast<size_t>(st) * kPiece);
#pragma unroll
          for (int kk = 0; kk < KP; ++kk) {
            const int kg = q * KP + kk;  // K-step within the tile: kmax part, then kmin part
            const uint64_t da = smem_desc(a0 + kk * 2 * kChunkBytes, kChunkBytes, 128);
            const uint64_t db = smem_desc(b0 + kg * 2 * (N * 16), N * 16, 128);
            tc_mma(tmem + static_cast<uint32_t>(acc * N), da, db, idesc, kg > 0 ? 1u : 0u);
          }
          tc_commit(&empty[st]);  // the stage is free once these MMAs have read it
          ++u;
          if (++st == stages) {
            st = 0;
            ++round;
          }
        }
        if (!ok) break;
        tc_commit(&accF[acc]);
        ++i;
      }
      // every MMA issued has completed before the tensor memory is released
      // (also after giving up half-way through a tile)
      if (u > 0) {
        tc_commit(drain);
        mbar_wait_bounded(drain, 0u, kWaitTriesTC);
      }
    }
  } else if (warp < 2 + kGroupWarps) {
    // ---------------- scan warps: query operands, C_b, stage release
    const int et = tid - 64;                   // 0 .. 127
    const int row = (warp & 3) * 32 + lane;    // the tile row (block) this thread owns
    const int Nq = G * Nd, Hq = Hkv * G;
    const int s_first = static_cast<int>(it.t0 / tps);
    const int s_last = it.t1 > it.t0 ? static_cast<int>((it.t1 - 1) / tps) : s_first - 1;
    int next_build = s_first, built = 0;
    // build {q+, q-} and Q of the next active segment into buffer built & 1
    constexpr int kItems = (N * CH + 32 * kGroupWarps - 1) / (32 * kGroupWarps);  // 16-byte query pieces per thread
    auto build_next = [&]() {
      while (next_build <= s_last && !it.active(next_build)) ++next_build;
      if (next_build > s_last) return;
      const int s = next_build, bq = built % kBBufs, qs = built & 1;  // operand buffer, Q / max slot
      const int bseq = s / Hkv, h = s % Hkv;
      uint8_t *B = sB + static_cast<size_t>(bq) * kBBytes;
      float *Q = sQ + qs * D;
      uint4 raw[kItems];
#pragma unroll
      for (int k = 0; k < kItems; ++k) {  // every load in flight before the first use
        const int item = et + k * 32 * kGroupWarps;
        if (item < N * CH) {
          const int n = item / CH, c = item % CH;
          const int j = min(n, Nq - 1), jd = j / G, g = j % G;
          raw[k] = __ldg(reinterpret_cast<const uint4 *>(
              qdraft + ((static_cast<int64_t>(bseq) * Nd + jd) * Hq + h * G + g) * D + c * 8));
        }
      }
      // the MMAs of the last segment that used this buffer have completed, and
      // the TMEM warps took the max_d Q_d of the last that used this slot (after
      // an abort the waits return at once; the outputs are then void anyway)
      if (built >= kBBufs)
        wait_or_abort(&bqE[bq], static_cast<uint32_t>((built / kBBufs) - 1) & 1u, abort_flag);
      if (built >= 2) wait_or_abort(&qmE[qs], static_cast<uint32_t>((built >> 1) - 1) & 1u, abort_flag);
      scan_barrier();  // every scan thread is done with this buffer's previous segment
#pragma unroll
      for (int k = 0; k < kItems; ++k) {
        const int item = et + k * 32 * kGroupWarps;
        if (item < N * CH) {
          const int n = item / CH, c = item % CH;
          const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
          uint32_t pos[4], neg[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t m = neg_halves(w4[e]);
            neg[e] = w4[e] & m;
            pos[e] = w4[e] & ~m;
          }
          *reinterpret_cast<uint4 *>(B + c * (N * 16) + n * 16) = make_uint4(pos[0], pos[1], pos[2], pos[3]);
          *reinterpret_cast<uint4 *>(B + (CH + c) * (N * 16) + n * 16) = make_uint4(neg[0], neg[1], neg[2], neg[3]);
        }
      }
      fence_proxy_async_smem();  // the tensor cores read B through the async proxy
      mbar_arrive(&bqF[bq]);
      scan_barrier();
      // Q_d = max over the query columns of |q_d|: a thread per pair of dims (non-
      // negative bf16 values order as integers; q+ and q- hold one of them each)
      for (int p = et; p < D / 2; p += 32 * kGroupWarps) {
        const int c = p / 4, e = p % 4;
        const uint32_t *colp = reinterpret_cast<const uint32_t *>(B + c * (N * 16)) + e;
        const uint32_t *coln = reinterpret_cast<const uint32_t *>(B + (CH + c) * (N * 16)) + e;
        uint32_t m = 0;
#pragma unroll 8
        for (int n = 0; n < N; ++n) m = __vmaxu2(m, (colp[n * 4] | coln[n * 4]) & 0x7FFF7FFFu);
        Q[2 * p] = bf16_lo(m);
        Q[2 * p + 1] = bf16_hi(m);
      }
      scan_barrier();  // Q is complete for every scan thread
      if (et == 0) {
        float qm = 0.0f;
        for (int d = 0; d < D; ++d) qm = fmaxf(qm, Q[d]);
        sQmax[qs] = qm;
        mbar_arrive(&qmF[qs]);
      }
      scan_barrier();
      ++next_build;
      ++built;
    };
    for (int k = 0; k < kBBufs; ++k) build_next();  // the first segments' operands
    // The group never leaves these loops early: after an abort every wait returns
    // at once and the work is skipped, so all four warps meet at the same named
    // barriers (inside build_next) whatever happened.
    if (wsum != nullptr) {
      // C_b <= max_d Q_d * wsum_b is formed by the TMEM warps themselves, so this
      // group only builds the active segments' query operands in turn (each build
      // waits until its buffer's previous segment is done with it)
      while (next_build <= s_last) build_next();
    } else {
      int64_t i = 0;         // tiles
      int st = 0;            // pieces % stages
      uint32_t round = 0;    // pieces / stages
      int seg_prev = -1, used = 0, bq = 0;
      for (it.begin(); it.valid(); it.advance()) {
        const int s = it.s;
        if (s != seg_prev) {
          if (seg_prev >= 0) build_next();  // the segment before is done: its buffer takes the next unbuilt one
          bq = used & 1;
          ++used;
          seg_prev = s;
        }
        const int base = it.j * kRows;
        const int rows = min(kRows, it.nc - base);
        // C_b: the summary values on the wrong side of zero, weighted by Q_d (kmax
        // half: |kmax| where kmax < 0; kmin half: kmin where kmin > 0), from the stages
        float C = 0.0f;
        {
#pragma unroll 1
          for (int q = 0; q < 2 * kPieces; ++q) {
            const int h = q / kPieces, c0 = (q % kPieces) * CP;
            const bool got = __all_sync(0xFFFFFFFFu, wait_or_abort(&full[st], round & 1u, abort_flag));
            if (got && row < rows) {
              const uint8_t *A = sA + static_cast<size_t>(st) * kPiece + row * 16;
              // fast test: any sign bit set among the kmax half (h = 0) / any clear among
              // the kmin half (h = 1)?  (-0 and +0 pass it too; their magnitude is 0)
              uint32_t acc_or = 0u, acc_and = 0xFFFFFFFFu;
#pragma unroll 8
              for (int c = 0; c < CP; ++c) {
                const uint4 x = *reinterpret_cast<const uint4 *>(A + c * kChunkBytes);
                acc_or |= x.x | x.y | x.z | x.w;
                acc_and &= x.x & x.y & x.z & x.w;
              }
              const bool wrong = h == 0 ? (acc_or & 0x80008000u) != 0u : (acc_and & 0x80008000u) != 0x80008000u;
              if (wrong) {  // the exact weighted sum
                const float *Q = sQ + bq * D;
                for (int c = 0; c < CP; ++c) {
                  const uint4 x = *reinterpret_cast<const uint4 *>(A + c * kChunkBytes);
                  const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
                  const float *Qc = Q + (c0 + c) * 8;
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const uint32_t m = neg_halves(xs[e]);
                    const uint32_t cw = h == 0 ? (xs[e] & m & 0x7FFF7FFFu) : (xs[e] & ~m);
                    C = fmaf(Qc[2 * e], bf16_lo(cw), C);
                    C = fmaf(Qc[2 * e + 1], bf16_hi(cw), C);
                  }
                }
              }
            }
            __syncwarp();
            if (got && lane == 0) mbar_arrive(&empty[st]);
            if (++st == stages) {
              st = 0;
              ++round;
            }
          }
        }
        const int cb = static_cast<int>(i % kNC);
        const bool room = i < kNC || __all_sync(0xFFFFFFFFu, wait_or_abort(&cE[cb], static_cast<uint32_t>((i / kNC) - 1) &
                                                                                       1u, abort_flag));
        if (room) {
          sC[cb * kRows + row] = C;
          mbar_arrive(&cF[cb]);
        }
        ++i;
      }
    }
  } else {
    // ---------------- TMEM warps: accumulator row -> max -> radius -> stores
    const int quad = warp & 3;                 // the TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    int64_t i = 0;
    int seg_cur = -1, used = 0;
    float qmax = 0.0f;  // max_d Q_d of the current segment
    const float gamma = 0x1p-12f, floor_r = 0x1p-110f;
    // this row's wrong-side sum in tile tt (0 past the candidates or without wsum)
    auto wsum_of = [&](const TileIter &w) -> float {
      if (wsum == nullptr || !w.valid()) return 0.0f;
      const int bb = w.j * kRows;
      return row < w.nc - bb ? __ldg(wsum + static_cast<int64_t>(w.s) * Nb_max + bb + row) : 0.0f;
    };
    TileIter cur = it;
    cur.begin();
    float ws = wsum_of(cur);  // loaded a tile ahead: its latency hides behind a whole tile
    while (cur.valid()) {
      TileIter nxt = cur;
      nxt.advance();
      const float ws_next = wsum_of(nxt);
      const int s = cur.s;
      const int base = cur.j * kRows;
      const int rows = min(kRows, cur.nc - base);
      const int acc = static_cast<int>(i % kNAcc);
      if (s != seg_cur) {  // take the segment's max_d Q_d and free its slot
        const int b = used & 1;
        if (!__all_sync(0xFFFFFFFFu, wait_or_abort(&qmF[b], static_cast<uint32_t>(used >> 1) & 1u, abort_flag)))
          break;
        qmax = sQmax[b];
        __syncwarp();
        if (lane == 0) mbar_arrive(&qmE[b]);
        ++used;
        seg_cur = s;
      }
      if (!__all_sync(0xFFFFFFFFu, wait_or_abort(&accF[acc], static_cast<uint32_t>(i / kNAcc) & 1u, abort_flag)))
        break;  // the whole warp leaves together
      tc_fence_after();
      float best = -FLT_MAX;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * N);
#pragma unroll
      for (int c0 = 0; c0 < N; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(taddr + c0, r);
        float m8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = max_nan(__uint_as_float(r[k]), __uint_as_float(r[k + 8]));
#pragma unroll
        for (int k = 0; k < 4; ++k) m8[k] = max_nan(m8[k], m8[k + 4]);
        best = max_nan(best, max_nan(max_nan(m8[0], m8[1]), max_nan(m8[2], m8[3])));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accE[acc]);
      float C = qmax * ws;  // with wsum: C_b <= max_d Q_d * wsum_b
      if (wsum == nullptr) {  // without: the scan warps' exact C_b
        const int cb = static_cast<int>(i % kNC);
        if (!__all_sync(0xFFFFFFFFu, wait_or_abort(&cF[cb], static_cast<uint32_t>(i / kNC) & 1u, abort_flag))) break;
        C = sC[cb * kRows + row];
        __syncwarp();
        if (lane == 0) mbar_arrive(&cE[cb]);
      }
      if (row < rows) {
        const bool nan = best != best;
        const int64_t o = static_cast<int64_t>(s) * Nb_max + base + row;
        scores[o] = best;
        radius[o] = nan ? __uint_as_float(0x7F800000u) : fmaf(gamma, fabsf(best) + 2.0f * C, floor_r);
      }
      ++i;
      cur = nxt;
      ws = ws_next;
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

// The summaries of one kind (kmin or kmax) as a 3-D tensor: x = 64 bf16 (8
// consecutive blocks of one 8-dim chunk, 128 bytes), y = Nb_max / 8 groups of 8
// blocks, z = S * CH chunks; one box = a piece (cp chunks of 128 blocks).
int make_summary_map(CUtensorMap *m, const uint16_t *base, int S, int CH, int cp, int Nb_max) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return -1;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(Nb_max / 8), static_cast<cuuint64_t>(S) * CH};
  const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(Nb_max) * 16};
  const cuuint32_t box[3] = {64, kRows / 8, static_cast<cuuint32_t>(cp)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? 0
             : -1;
}

template <int N, int CH>
cudaError_t launch_tc(const uint16_t *kmin, const uint16_t *kmax, const float *wsum, int Nb_max,
                      const uint16_t *qdraft, int B, int Hkv, int G, int Nd, const int32_t *seq_len, int W,
                      float *scores, float *radius, int32_t *status, cudaStream_t st) {
  constexpr int kCP = CH / pieces<N, CH>();  // chunks per piece
  constexpr size_t kPiece = static_cast<size_t>(kCP) * kChunkBytes;
  const int S = B * Hkv;
  const int ncand = Nb_max - W;
  if (ncand <= 0) return cudaSuccess;  // no candidate can exist
  const int tps = (ncand + kRows - 1) / kRows;
  // A tile's rows read by the tensor copies may run past Nb_max (zero-filled);
  // the tensor view needs whole groups of 8 blocks, else 16-byte bulk copies
  CUtensorMap tmx{}, tmn{};
  const bool use_tma = Nb_max % 8 == 0 && make_summary_map(&tmx, kmax, S, CH, kCP, Nb_max) == 0 &&
                       make_summary_map(&tmn, kmin, S, CH, kCP, Nb_max) == 0;
  const size_t fixed = fixed_smem<N, CH>();
  const int stages = static_cast<int>(std::min<size_t>(kMaxStages, (kSmemCap - fixed) / kPiece));
  if (stages < 2) return cudaErrorInvalidValue;
  const size_t smem = fixed + stages * kPiece;
  int sms = 0, per_sm = 0;
  cudaError_t e = launch_geometry(reinterpret_cast<const void *>(k_score_tc<N, CH>), kThreadsTC, smem, &sms, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t T = static_cast<int64_t>(S) * tps;
  // Two CTAs per SM, the tiles split evenly.  When every segment spans four or
  // more CTAs' shares, the CTAs are instead aligned to segments (k per segment,
  // 4 <= k <= two per SM / S): each CTA then builds one query operand, where
  // short shares across segment boundaries spend more in rebuilds than a few
  // idle MMA lanes cost (64 segments: 15.4 -> 15.0 us; with k = 1 or 2 the
  // lanes left idle cost more, 48.3 -> 52.6 us at 256 segments)
  int64_t grid = static_cast<int64_t>(kCtasPerSm) * sms;
  if (grid / S >= 4) grid = static_cast<int64_t>(S) * (grid / S);
  grid = std::min<int64_t>(grid, T);
  LaunchCfg lc(dim3(static_cast<unsigned>(grid)), dim3(kThreadsTC), smem, st);
  return cudaLaunchKernelEx(&lc.cfg, k_score_tc<N, CH>, tmx, tmn, use_tma, kmin, kmax, wsum, Nb_max, qdraft, S,
                            Hkv, G, Nd, seq_len, W, scores, radius, status, tps, stages);
}

template <int CH>
cudaError_t launch_tc_n(const uint16_t *kmin, const uint16_t *kmax, const float *wsum, int Nb_max,
                        const uint16_t *qdraft, int B, int Hkv, int G, int Nd, const int32_t *seq_len, int W,
                        float *scores, float *radius, int32_t *status, cudaStream_t st) {
  const int Nq = G * Nd;
#define OASIS_TC_CASE(NN)                                                                                       \
  if (Nq <= NN)                                                                                                  \
    return launch_tc<NN, CH>(kmin, kmax, wsum, Nb_max, qdraft, B, Hkv, G, Nd, seq_len, W, scores, radius, status, \
                             st);
  OASIS_TC_CASE(16)
  OASIS_TC_CASE(32)
  OASIS_TC_CASE(48)
  OASIS_TC_CASE(64)
#undef OASIS_TC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_score_blocks_tc(const uint16_t *kmin, const uint16_t *kmax, const float *wsum, int Nb_max,
                                   const uint16_t *qdraft, int B, int Hkv, int G, int Nd, int D,
                                   const int32_t *seq_len, int W, float *scores, float *radius, int32_t *status,
                                   cudaStream_t st) {
  if (D == 128)
    return launch_tc_n<16>(kmin, kmax, wsum, Nb_max, qdraft, B, Hkv, G, Nd, seq_len, W, scores, radius, status, st);
  return launch_tc_n<8>(kmin, kmax, wsum, Nb_max, qdraft, B, Hkv, G, Nd, seq_len, W, scores, radius, status, st);
}

}  // namespace oasis
