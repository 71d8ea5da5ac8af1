// Sparse paged decode attention on the tcgen05 tensor cores.
//
// OasisKV paper review (xllm-io), §3 Fig. 5: the foreground forward pass runs
// sparse attention of the true query over the working set resident in HBM;
// §4 / Fig. 9: each KV head addresses its own resident blocks through the
// head-wise mapping.  For query head h*G + g of sequence b:
//     out = sum_i softmax_i(scale * q . k_i) v_i
// over the valid tokens of the slots whose table entry is >= 0 (the same
// operation as the mma.sync kernels of attention.cu, same outputs and status).
//
// Shape: d_h 128, up to 16 query heads per KV head.  A segment (one KV head of
// one sequence) is split over a cluster of CL CTAs (slot k goes to CTA k % CL).
// A CTA lists its non-empty slots, then walks them in tiles of 8 slots = 128
// tokens:
//   S^T[128 tokens x 16 heads] = K[128 x 128] . Q^T          (one tcgen05 MMA chain, M 128, N 16)
//   online softmax over the tile's tokens, per head, in the log2 domain
//   O_t^T[128 dims x 16 heads] = V^T[128 x 128] . P^T         (P^T as bf16 hi + lo parts)
// so the tensor cores carry both products and the threads only the softmax.
// Operands in shared memory:
//   keys / values of a tile: 8 slots x 16 rows, one 2-D TMA copy per slot and
//     64-dim half into [half][128 rows][128 B] with the 128-byte swizzle; the
//     keys are the K-major A operand of the first product (8-row groups 1 KiB
//     apart), the values the MN-major A operand of the second (64-dim groups
//     16 KiB apart, 8-token groups 1 KiB apart);
//   Q^T and P^T: no-swizzle core matrices of 8 rows x 16 bytes, [k-group][n-group]
//     (k-groups 256 B apart, n-groups 128 B apart); Q^T K-major (rows = heads),
//     P^T MN-major (rows = tokens, 8 heads per 16 bytes).
// Roles (warp-specialised, mbarrier hand-offs, every wait bounded):
//   warp 0, one lane - the copies: keys, then values, of each tile through a
//                      ring of 32 KiB stages;
//   warp 1, one lane - the MMAs, as two streams polled without blocking: S of a
//                      tile once its keys have landed, P.V of a tile once its
//                      P^T is written, each independent of the other (a lane
//                      that waited for the next keys before issuing P.V would
//                      hold the values, and with them the next copy, for a
//                      whole memory latency per tile); owns the tensor memory;
//   warps 2-5        - one tensor-memory lane each: token row of S for the
//                      softmax, dim row of O for the output.  Per tile: the
//                      head maxima over the 128 rows (a transposing warp
//                      butterfly, then the four warps through shared memory),
//                      p = 2^(x - m), P^T written for the MMA, and the previous
//                      tile's O_t folded into registers as o = o * c + O_t, c
//                      the rescale factor of the running maxima.  Each thread
//                      also keeps a per-row partial of the softmax sums.
// Two CTAs fit an SM.  The cluster merges its CTAs' (m, l, o) through
// distributed shared memory as the mma.sync kernels do; one CTA writes out and
// lse directly.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cfloat>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace oasis {
namespace {

constexpr int kD = 128;                                // head dim of this kernel
constexpr int kTileSlots = 8;                          // slots per tile
constexpr int kTileRows = kTileSlots * kBlockTokens;   // 128 tokens: MMA M of S^T
constexpr int kN = 16;                                 // query heads per KV head, padded: MMA N
constexpr int kSoftWarps = 4;
constexpr int kThreadsA = 32 * (2 + kSoftWarps);
constexpr uint32_t kStageBytes = kTileRows * kD * 2;   // the keys or the values of a tile: 32 KiB
constexpr uint32_t kHalfBytes = kStageBytes / 2;       // one 64-dim half: 128 rows x 128 B
constexpr uint32_t kSlotHalfBytes = kBlockTokens * 128;  // one slot's rows of a half: 2 KiB
constexpr uint32_t kQBytes = kN * kD * 2;              // Q^T: 4 KiB
constexpr uint32_t kPBytes = kTileRows * kN * 2;       // one part of P^T: 4 KiB
constexpr uint32_t kTmemColsA = 64;                    // S: 2 x 16 columns, O: 2 x 16
constexpr uint32_t kWaitTriesA = 1u << 22;             // bounded mbarrier polls (far beyond any real copy or MMA)
constexpr uint32_t kIdlePolls = 1u << 26;              // MMA lane: non-blocking polls without progress
constexpr int kMinStagesA = 2, kMaxStagesA = 3;
constexpr int kMaxClusterA = 4;
constexpr size_t kSmemCapA = (228 * 1024) / 2 - 1024;  // two CTAs per SM
constexpr int kNumBarsA = 2 * kMaxStagesA + 11;
constexpr float kLn2A = 0.69314718055994530942f;

// Shared-memory plan: offsets from a 1024-aligned base.
struct AttnPlan {
  uint32_t q, p, red, redl, bars, misc, list, end;
};
__host__ __device__ __forceinline__ AttnPlan attn_plan(int stages, int list_cap) {
  AttnPlan P;
  P.q = static_cast<uint32_t>(stages) * kStageBytes;
  P.p = P.q + kQBytes;
  P.red = P.p + 2 * kPBytes;             // float [2][kSoftWarps][kN]: per-warp tile maxima
  P.redl = P.red + 2 * kSoftWarps * kN * 4;  // float [kSoftWarps][kN]: per-warp softmax sums
  P.bars = P.redl + kSoftWarps * kN * 4;
  P.misc = P.bars + kNumBarsA * 8;       // tmem base, abort flag, list length
  P.list = P.misc + 16;
  P.end = P.list + 4 * static_cast<uint32_t>(list_cap);
  return P;
}

// ---- tcgen05 / TMEM primitives (inline PTX) ---------------------------------
// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets in 16-byte units, descriptor version bit 46, swizzle mode in bits
// 61-63 (0 none, 2 the 128-byte swizzle).
__device__ __forceinline__ uint64_t mdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint64_t swz) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
         (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46) | (swz << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulator (bit 4), bf16 A and B
// (bits 7, 10), A / B MN-major when set (bits 15, 16), N >> 3 at bit 17,
// M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_attn(bool mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (mn_major ? (1u << 15) | (1u << 16) : 0u) |
         (static_cast<uint32_t>(kN >> 3) << 17) | (static_cast<uint32_t>(kTileRows >> 4) << 24);
}
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 16 consecutive fp32 columns of this thread's TMEM lane, waited for.
__device__ __forceinline__ void tmem_load16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}
__device__ __forceinline__ void arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void soft_barrier() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kSoftWarps) : "memory"); }
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}
// {lo, hi} -> bf16x2 with `lo` in the low half (round to nearest even)
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Non-blocking test of phase `parity` of `bar`.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait that also gives up once another role has given up.
__device__ __forceinline__ bool wait_or_give_up(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
  for (uint32_t k = 0; k < kWaitTriesA; ++k) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

// 16 per-lane values reduced (max or sum) over the 32 lanes of a warp, with the
// result transposed: lane L returns value L >> 1.  Each step keeps half of the
// values and trades the other half with the partner lane.
template <bool kMax>
__device__ __forceinline__ float warp_reduce16(const float (&v)[16], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float a[8], b[4], c[2];
  const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    a[i] = op(u16 ? v[i + 8] : v[i], __shfl_xor_sync(0xFFFFFFFFu, u16 ? v[i] : v[i + 8], 16));
#pragma unroll
  for (int i = 0; i < 4; ++i)
    b[i] = op(u8 ? a[i + 4] : a[i], __shfl_xor_sync(0xFFFFFFFFu, u8 ? a[i] : a[i + 4], 8));
#pragma unroll
  for (int i = 0; i < 2; ++i)
    c[i] = op(u4 ? b[i + 2] : b[i], __shfl_xor_sync(0xFFFFFFFFu, u4 ? b[i] : b[i + 2], 4));
  float d = op(u2 ? c[1] : c[0], __shfl_xor_sync(0xFFFFFFFFu, u2 ? c[0] : c[1], 2));
  return op(d, __shfl_xor_sync(0xFFFFFFFFu, d, 1));
}

__global__ void __launch_bounds__(kThreadsA, 2)
    k_attn_tc(const __grid_constant__ CUtensorMap tmap, const uint16_t *__restrict__ q,
              const int32_t *__restrict__ table, int slots, const int32_t *__restrict__ seq_len, int Hkv, int G,
              float scale_log2, float *__restrict__ out, float *__restrict__ lse, int32_t *status, int stages,
              int list_cap) {
  extern __shared__ unsigned char sm_raw[];
  unsigned char *sm = sm_raw + ((1024u - (smem_addr(sm_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(sm);
  const AttnPlan Pl = attn_plan(stages, list_cap);
  cg::cluster_group cluster = cg::this_cluster();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int s = blockIdx.y;
  const int bseq = s / Hkv, hk = s % Hkv;
  const int Hq = Hkv * G;

  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Pl.bars);
  uint64_t *full = bars, *empty = bars + kMaxStagesA;
  uint64_t *sF = bars + 2 * kMaxStagesA, *sE = sF + 2, *pF = sE + 2, *pE = pF + 1, *oF = pE + 1, *oE = oF + 2;
  uint64_t *drain = oE + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Pl.misc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + Pl.misc + 4);
  int *count_slot = reinterpret_cast<int *>(sm + Pl.misc + 8);
  int32_t *list = reinterpret_cast<int32_t *>(sm + Pl.list);

  int L = seq_len[bseq];
  if (L < 0) {
    if (tid == 0 && rank == 0 && hk == 0) report(status, OASIS_STATUS_SEQ_LEN);
    L = 0;
  }
  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);  // the MMAs' commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sF[i], 1);
      mbar_init(&sE[i], kSoftWarps);
      mbar_init(&oF[i], 1);
      mbar_init(&oE[i], kSoftWarps);
    }
    mbar_init(pF, kSoftWarps);
    mbar_init(pE, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kTmemColsA)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  } else if (warp == 0) {
    // this CTA's non-empty slots (slot k of the segment goes to CTA k % CL), as
    // (slot << 5 | valid tokens)
    const int nk = slots > rank ? (slots - rank + CL - 1) / CL : 0;
    const int32_t *trow = table + static_cast<int64_t>(s) * slots;
    int count = 0;
    for (int base = 0; base < nk; base += 32) {
      const int k = base + lane;
      int nv = 0, slot = 0;
      if (k < nk) {
        slot = rank + CL * k;
        const int blk = trow[slot];
        const int64_t n = blk < 0 ? 0 : static_cast<int64_t>(L) - static_cast<int64_t>(kBlockTokens) * blk;
        nv = n <= 0 ? 0 : (n >= kBlockTokens ? kBlockTokens : static_cast<int>(n));
      }
      const unsigned mk = __ballot_sync(0xFFFFFFFFu, nv > 0);
      if (nv > 0) list[count + __popc(mk & ((1u << lane) - 1u))] = (slot << 5) | nv;
      count += __popc(mk);
    }
    if (lane == 0) *count_slot = count;
  }
  // Q^T operand: head n (rows, zero past G), dims c*8 .. c*8+7 per 16-byte piece
  for (int item = tid; item < kN * (kD / 8); item += kThreadsA) {
    const int n = item / (kD / 8), c = item % (kD / 8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < G)
      v = __ldg(reinterpret_cast<const uint4 *>(q + (static_cast<int64_t>(bseq) * Hq + hk * G + n) * kD + c * 8));
    *reinterpret_cast<uint4 *>(sm + Pl.q + c * 256 + (n >> 3) * 128 + (n & 7) * 16) = v;
  }
  fence_proxy_async_smem();  // the tensor cores read Q^T through the async proxy
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int count = *count_slot;
  const int ntile = (count + kTileSlots - 1) / kTileSlots;

  // the partial results of the tiles (softmax warps; the final merge reads them)
  float m[kN], l[kN], o[kN];

  if (warp == 0) {
    // ---------------- copies: keys of tile t, then its values, stage by stage
    if (lane == 0) {
      const int row_base = s * slots;
      int issued = 0, st = 0;
      uint32_t round = 0;
      for (int u = 0; u < 2 * ntile; ++u) {
        if (u >= stages && !wait_or_give_up(&empty[st], (round - 1u) & 1u, abort_flag)) break;
        const int t = u >> 1, kind = u & 1;
        mbar_arrive_expect_tx(&full[st], kStageBytes);
        const uint32_t dst = sbase + static_cast<uint32_t>(st) * kStageBytes;
#pragma unroll 1
        for (int j = 0; j < kTileSlots; ++j) {
          // past the list: the last listed slot again (its rows are masked)
          const int e = min(t * kTileSlots + j, count - 1);
          const int y = (row_base + (list[e] >> 5)) * 32 + kind * kBlockTokens;
          tma_2d(dst + j * kSlotHalfBytes, &tmap, 0, y, &full[st]);
          tma_2d(dst + kHalfBytes + j * kSlotHalfBytes, &tmap, 64, y, &full[st]);
        }
        ++issued;
        if (++st == stages) {
          st = 0;
          ++round;
        }
      }
      // never leave with copies in flight
      for (int k = max(0, issued - stages); k < issued; ++k)
        mbar_wait_bounded(&full[k % stages], static_cast<uint32_t>(k / stages) & 1u, kWaitTriesA);
    }
  } else if (warp == 1) {
    // ---------------- MMAs
    if (lane == 0) {
      constexpr uint32_t idS = idesc_attn(false), idPV = idesc_attn(true);
      const uint32_t sq = sbase + Pl.q, sp = sbase + Pl.p;
      int mmas = 0;
      // Two streams of MMAs, each issued as soon as its inputs are ready: S of
      // tile ts (its keys have landed, its S buffer is free) and P.V of tile tp
      // (its P^T is written, its values have landed, its O buffer is free).
      // Neither waits for the other, so the values of tile tp are released (and
      // the next keys copied) as soon as the softmax of tile tp is done.
      // A parity test tells phases apart only modulo 2, so item u's copy is
      // tested only once the item before it in the same stage (u - stages) has
      // been taken by an MMA: its copy has then landed, and the stage's barrier
      // is at most one phase behind.  (Item 2t = the keys of tile t, 2t + 1 its
      // values.)
      int ts = 0, tp = 0;
      auto taken = [&](int v) { return v < 0 || ((v & 1) ? (v >> 1) < tp : (v >> 1) < ts); };
      uint32_t idle = 0;
      while (tp < ntile) {
        bool did = false;
        if (ts < ntile && taken(2 * ts - stages)) {
          const int u = 2 * ts, st = u % stages;
          if (mbar_test(&full[st], static_cast<uint32_t>(u / stages) & 1u) &&
              (ts < 2 || mbar_test(&sE[ts & 1], static_cast<uint32_t>((ts >> 1) - 1) & 1u))) {
            tmem_fence_after();
            const uint32_t a0 = sbase + static_cast<uint32_t>(st) * kStageBytes;
#pragma unroll
            for (int k = 0; k < kD / 16; ++k) {  // 16 dims per MMA: 32 bytes into the swizzled row
              const uint64_t da = mdesc(a0 + (k >> 2) * kHalfBytes + (k & 3) * 32, 16, 1024, 2);
              mma_f16(tmem + static_cast<uint32_t>(ts & 1) * kN, da, mdesc(sq + k * 512, 256, 128, 0), idS,
                      k > 0 ? 1u : 0u);
            }
            mma_commit(&empty[st]);
            mma_commit(&sF[ts & 1]);
            ++mmas;
            ++ts;
            did = true;
          }
        }
        if (tp < ts && taken(2 * tp + 1 - stages)) {
          const int u = 2 * tp + 1, st = u % stages;
          if (mbar_test(pF, static_cast<uint32_t>(tp) & 1u) &&
              mbar_test(&full[st], static_cast<uint32_t>(u / stages) & 1u) &&
              (tp < 2 || mbar_test(&oE[tp & 1], static_cast<uint32_t>((tp >> 1) - 1) & 1u))) {
            tmem_fence_after();
            const uint32_t a0 = sbase + static_cast<uint32_t>(st) * kStageBytes;
            const uint32_t dcol = tmem + 32u + static_cast<uint32_t>(tp & 1) * kN;
#pragma unroll
            for (int j = 0; j < kTileRows / 16; ++j) {  // 16 tokens per MMA
              const uint64_t da = mdesc(a0 + j * 2048, kHalfBytes, 1024, 2);
              mma_f16(dcol, da, mdesc(sp + j * 512, 256, 128, 0), idPV, j > 0 ? 1u : 0u);
              mma_f16(dcol, da, mdesc(sp + kPBytes + j * 512, 256, 128, 0), idPV, 1u);
            }
            mma_commit(&empty[st]);
            mma_commit(&oF[tp & 1]);
            mma_commit(pE);
            ++mmas;
            ++tp;
            did = true;
          }
        }
        if (did) {
          idle = 0;
        } else if (++idle > kIdlePolls || *abort_flag) {
          *abort_flag = 1;
          break;
        }
      }
      // every MMA issued has completed before the tensor memory is released
      if (mmas > 0) {
        mma_commit(drain);
        mbar_wait_bounded(drain, 0u, kWaitTriesA);
      }
    }
  } else {
    // ---------------- softmax warps: TMEM lane `row` (a token of S, a dim of O)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    float *red = reinterpret_cast<float *>(sm + Pl.red);
    float c_prev[kN];
#pragma unroll
    for (int h = 0; h < kN; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.0f;  // this row's share of the sums
      o[h] = 0.0f;
      c_prev[h] = 1.0f;
    }
    // o <- o * c_prev + O_t (rows = dims); after an abort every wait returns at
    // once, and the group still meets at every named barrier
    auto fold_o = [&](int t) {
      __all_sync(0xFFFFFFFFu, wait_or_give_up(&oF[t & 1], static_cast<uint32_t>(t >> 1) & 1u, abort_flag));
      tmem_fence_after();
      uint32_t r[16];
      tmem_load16(tl + 32u + static_cast<uint32_t>(t & 1) * kN, r);
      tmem_fence_before();
      __syncwarp();
      if (lane == 0) arrive(&oE[t & 1]);
#pragma unroll
      for (int h = 0; h < kN; ++h) o[h] = fmaf(o[h], c_prev[h], __uint_as_float(r[h]));
    };
    for (int t = 0; t < ntile; ++t) {
      __all_sync(0xFFFFFFFFu, wait_or_give_up(&sF[t & 1], static_cast<uint32_t>(t >> 1) & 1u, abort_flag));
      tmem_fence_after();
      uint32_t r[16];
      tmem_load16(tl + static_cast<uint32_t>(t & 1) * kN, r);
      tmem_fence_before();
      __syncwarp();
      if (lane == 0) arrive(&sE[t & 1]);
      const int e = t * kTileSlots + (row >> 4);
      const int ent = e < count ? list[e] : 0;
      const bool valid = (row & 15) < (ent & 31);
      float x[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h) x[h] = valid ? __uint_as_float(r[h]) * scale_log2 : -INFINITY;
      // tile maxima per head: this warp's 32 rows, then the four warps
      const float wm = warp_reduce16<true>(x, lane);
      float *rb = red + (t & 1) * kSoftWarps * kN;
      if ((lane & 1) == 0) rb[quad * kN + (lane >> 1)] = wm;
      soft_barrier();
      float c[kN], p[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        const float tmx = fmaxf(fmaxf(rb[h], rb[kN + h]), fmaxf(rb[2 * kN + h], rb[3 * kN + h]));
        const float mn = fmaxf(m[h], tmx);
        const bool none = mn == -INFINITY;  // no valid token of this head yet
        c[h] = none ? 1.0f : exp2f(m[h] - mn);
        p[h] = none ? 0.0f : exp2f(x[h] - mn);
        m[h] = mn;
        l[h] = fmaf(l[h], c[h], p[h]);
      }
      uint32_t hi[kN / 2], lo[kN / 2];
#pragma unroll
      for (int i = 0; i < kN / 2; ++i) {
        hi[i] = bf16x2(p[2 * i], p[2 * i + 1]);
        lo[i] = bf16x2(p[2 * i] - bf16_lo(hi[i]), p[2 * i + 1] - bf16_hi(hi[i]));
      }
      // P^T rows: token `row` = row (row & 7) of k-group row >> 3; heads 0-7, then 8-15
      if (t >= 1)
        __all_sync(0xFFFFFFFFu, wait_or_give_up(pE, static_cast<uint32_t>(t - 1) & 1u, abort_flag));
      unsigned char *P = sm + Pl.p + (row >> 3) * 256 + (row & 7) * 16;
      *reinterpret_cast<uint4 *>(P) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4 *>(P + 128) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
      *reinterpret_cast<uint4 *>(P + kPBytes) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<uint4 *>(P + kPBytes + 128) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) arrive(pF);
      if (t >= 1) fold_o(t - 1);
#pragma unroll
      for (int h = 0; h < kN; ++h) c_prev[h] = c[h];
    }
    if (ntile > 0) fold_o(ntile - 1);
    // softmax sums over the 128 rows
    const float ws = warp_reduce16<false>(l, lane);
    float *redl = reinterpret_cast<float *>(sm + Pl.redl);
    if ((lane & 1) == 0) redl[quad * kN + (lane >> 1)] = ws;
    soft_barrier();
#pragma unroll
    for (int h = 0; h < kN; ++h) l[h] = (redl[h] + redl[kN + h]) + (redl[2 * kN + h] + redl[3 * kN + h]);
    if (CL == 1) {
      const int64_t row0 = static_cast<int64_t>(bseq) * Hq + hk * G;
#pragma unroll
      for (int h = 0; h < kN; ++h)
        if (h < G) out[(row0 + h) * kD + row] = l[h] > 0.0f ? o[h] / l[h] : 0.0f;
      if (lse != nullptr && row < G) {
        float mh = 0.0f, lh = 0.0f;
#pragma unroll
        for (int h = 0; h < kN; ++h)
          if (h == row) {
            mh = m[h];
            lh = l[h];
          }
        lse[row0 + row] = lh > 0.0f ? (mh + log2f(lh)) * kLn2A : -INFINITY;
      }
    }
  }

  tmem_fence_before();
  __syncthreads();  // every role is done: no copy or MMA is in flight
  if (*abort_flag && tid == 0) report(status, OASIS_STATUS_TIMEOUT);
  if (warp == 1) {
    tmem_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemColsA) : "memory");
  }
  if (CL > 1) {
    // cluster merge: every CTA's (m, l, o) in its ring, then each CTA combines a
    // 1/CL share of the outputs from all of them
    float *cm = reinterpret_cast<float *>(sm), *cl = cm + kN, *co = cl + kN;  // co: [kN][kD]
    if (warp >= 2) {
      const int row = (warp & 3) * 32 + lane;
#pragma unroll
      for (int h = 0; h < kN; ++h) co[h * kD + row] = o[h];
      if (row < kN) {
        float mh = 0.0f, lh = 0.0f;
#pragma unroll
        for (int h = 0; h < kN; ++h)
          if (h == row) {
            mh = m[h];
            lh = l[h];
          }
        cm[row] = mh;
        cl[row] = lh;
      }
    }
    cluster.sync();
    const int n_out = G * kD, per = (n_out + CL - 1) / CL;
    const int e1 = min(n_out, (rank + 1) * per);
    for (int idx = rank * per + tid; idx < e1; idx += kThreadsA) {
      const int qc = idx / kD, d = idx % kD;
      float mr[kMaxClusterA], lr[kMaxClusterA], orr[kMaxClusterA];
#pragma unroll
      for (int r = 0; r < kMaxClusterA; ++r) {
        if (r < CL) {
          mr[r] = cluster.map_shared_rank(cm, r)[qc];
          lr[r] = cluster.map_shared_rank(cl, r)[qc];
          orr[r] = cluster.map_shared_rank(co, r)[qc * kD + d];
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < kMaxClusterA; ++r)
        if (r < CL) M = fmaxf(M, mr[r]);
      float acc = 0.0f, ls = 0.0f;
      if (M > -INFINITY) {
#pragma unroll
        for (int r = 0; r < kMaxClusterA; ++r) {
          if (r < CL) {
            const float f = exp2f(mr[r] - M);
            acc += f * orr[r];
            ls += f * lr[r];
          }
        }
      }
      const int64_t orow = static_cast<int64_t>(bseq) * Hq + hk * G + qc;
      out[orow * kD + d] = ls > 0.0f ? acc / ls : 0.0f;
      if (d == 0 && lse != nullptr) lse[orow] = ls > 0.0f ? (M + log2f(ls)) * kLn2A : -INFINITY;
    }
    cluster.sync();  // no CTA leaves while another may still read its shared memory
  }
}

}  // namespace

// The slot pool as rows of 128 bf16 (16 key rows, then 16 value rows per
// slot), read in boxes of 64 dims x 16 rows (one slot's keys or values of one
// half) with the 128-byte swizzle.
static cudaError_t make_pool_map16(CUtensorMap *tmap, const uint16_t *pool, int S, int slots) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(S) * slots * 32};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBlockTokens)};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(pool), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

bool attn_tc_supports(int G, int D) { return D == kD && G >= 1 && G <= kN; }

cudaError_t launch_attn_tc(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots,
                           const int32_t *seq_len, int B, int Hkv, int G, int D, float scale, float *out, float *lse,
                           int32_t *status, cudaStream_t st) {
  if (!attn_tc_supports(G, D)) return cudaErrorInvalidValue;
  const int S = B * Hkv;
  int sms = 0, per_sm = 0;
  cudaError_t e = launch_geometry(reinterpret_cast<const void *>(k_attn_tc), kThreadsA, kSmemCapA, &sms, &per_sm);
  if (e != cudaSuccess) return e;
  // about two CTAs per SM in all
  int CL = static_cast<int>(std::min<int64_t>(kMaxClusterA, std::max<int64_t>(1, 2 * static_cast<int64_t>(sms) / S)));
  CL = std::min(CL, slots);
  // the list: this CTA's slots, rounded up to whole tiles
  const int per_cta = (slots + CL - 1) / CL;
  const int list_cap = (per_cta + kTileSlots - 1) / kTileSlots * kTileSlots;
  int stages = kMaxStagesA;
  while (stages >= kMinStagesA && attn_plan(stages, list_cap).end + 1024 > kSmemCapA) --stages;
  if (stages < kMinStagesA) return cudaErrorInvalidValue;
  const size_t smem = attn_plan(stages, list_cap).end + 1024;  // + slack for the 1024-byte alignment
  CUtensorMap tmap;
  e = make_pool_map16(&tmap, pool, S, slots);
  if (e != cudaSuccess) return e;
  e = launch_geometry(reinterpret_cast<const void *>(k_attn_tc), kThreadsA, smem, &sms, &per_sm);
  if (e != cudaSuccess) return e;
  LaunchCfg lc(dim3(static_cast<unsigned>(CL), static_cast<unsigned>(S)), dim3(kThreadsA), smem, st);
  cudaLaunchAttribute cl;
  cl.id = cudaLaunchAttributeClusterDimension;
  cl.val.clusterDim.x = static_cast<unsigned>(CL);
  cl.val.clusterDim.y = 1;
  cl.val.clusterDim.z = 1;
  lc.add(cl);
  const float scale_log2 = scale * 1.4426950408889634f;
  return cudaLaunchKernelEx(&lc.cfg, k_attn_tc, tmap, q, table, slots, seq_len, Hkv, G, scale_log2, out, lse, status,
                            stages, list_cap);
}

}  // namespace oasis
