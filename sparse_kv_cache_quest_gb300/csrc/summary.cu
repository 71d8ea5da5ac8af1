// Min/max key summaries per 16-token block (Quest-style compressed key cache).
//
// OasisKV paper review (xllm-io), §3 component table "Compressed Key Cache":
// every logical block keeps a per-dimension min/max of its keys, 1/16 of the
// full KV; §5: compressed keys are updated during decode.
//
// One thread per (segment, block, 8-dim chunk), over a flat grid: it issues
// the 16-byte loads of the chunk from all valid token rows at once
// (consecutive threads read consecutive chunks of a row, so a warp reads whole
// 256-byte rows) and writes 16 bytes to kmin and kmax in the chunk-major
// layout [S][D/8][Nb_max][8].
//
// Optionally (wsum != NULL) each block also gets the sum over its dims of the
// summary values on the "wrong" side of zero - |kmax_d| where kmax_d < 0, kmin_d
// where kmin_d > 0 - rounded up: the tensor-core scoring bounds its error with
// it.  The 16 (or 8) chunk threads of a block are consecutive lanes of one warp
// and add their parts in a fixed butterfly order.
//
// min/max use the IEEE 754-2019 total order of non-NaN values (-0 below +0):
// each bf16 bit pattern u maps to the 16-bit key u | 0x8000 (u >= +0) or ~u
// (u negative), which is monotone in value, so unsigned min/max of keys picks
// the IEEE minimum/maximum exactly.  Two halves of a 32-bit word are handled
// at once with the SIMD-within-a-word intrinsics __vminu2 / __vmaxu2.
#include "common.cuh"

namespace oasis {
namespace {

__device__ __forceinline__ uint32_t to_key2(uint32_t w) {
  const uint32_t neg = (w >> 15) & 0x00010001u;
  return w ^ ((neg * 0x7FFFu) | 0x80008000u);
}
__device__ __forceinline__ uint32_t from_key2(uint32_t k) {
  const uint32_t neg = ((~k) >> 15) & 0x00010001u;
  return k ^ ((neg * 0x7FFFu) | 0x80008000u);
}

__global__ void __launch_bounds__(256) k_build_summary(const uint16_t *__restrict__ k, int64_t seg_stride,
                                                       int64_t blk_stride, int64_t tok_stride, int Hkv, int D,
                                                       const int32_t *__restrict__ seq_len, int blk_begin,
                                                       int blk_count, int S, uint16_t *__restrict__ kmin,
                                                       uint16_t *__restrict__ kmax, float *__restrict__ wsum,
                                                       int Nb_max, int32_t *status) {
  const int chunks = D >> 3;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // every early return below takes a block's chunk threads (an aligned group of
  // `chunks` lanes) together, so the group's shuffles see all of their lanes
  if (item >= static_cast<int64_t>(S) * blk_count * chunks) return;
  const int c = static_cast<int>(item % chunks);
  const int64_t sj = item / chunks;
  const int j = static_cast<int>(sj % blk_count);
  const int s = static_cast<int>(sj / blk_count);
  const int L = load_len(seq_len, s / Hkv, Nb_max * kBlockTokens, status, j == 0 && c == 0 && (s % Hkv) == 0);
  const int b = blk_begin + j;
  const int nvalid = min(kBlockTokens, L - kBlockTokens * b);
  if (nvalid <= 0) return;

  const uint16_t *p = k + s * seg_stride + j * blk_stride + c * 8;
  uint4 v[kBlockTokens];
#pragma unroll
  for (int t = 0; t < kBlockTokens; ++t)  // all loads in flight at once
    if (t < nvalid) v[t] = __ldg(reinterpret_cast<const uint4 *>(p + t * tok_stride));
  uint4 lo = make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
  uint4 hi = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int t = 0; t < kBlockTokens; ++t) {
    if (t < nvalid) {
      const uint32_t a = to_key2(v[t].x), bb = to_key2(v[t].y), cc = to_key2(v[t].z), dd = to_key2(v[t].w);
      lo.x = __vminu2(lo.x, a);
      lo.y = __vminu2(lo.y, bb);
      lo.z = __vminu2(lo.z, cc);
      lo.w = __vminu2(lo.w, dd);
      hi.x = __vmaxu2(hi.x, a);
      hi.y = __vmaxu2(hi.y, bb);
      hi.z = __vmaxu2(hi.z, cc);
      hi.w = __vmaxu2(hi.w, dd);
    }
  }
  const int64_t o = ((static_cast<int64_t>(s) * chunks + c) * Nb_max + b) * 8;
  const uint4 mn = make_uint4(from_key2(lo.x), from_key2(lo.y), from_key2(lo.z), from_key2(lo.w));
  const uint4 mx = make_uint4(from_key2(hi.x), from_key2(hi.y), from_key2(hi.z), from_key2(hi.w));
  *reinterpret_cast<uint4 *>(kmin + o) = mn;
  *reinterpret_cast<uint4 *>(kmax + o) = mx;
  if (wsum != nullptr) {
    const uint32_t xs[4] = {mx.x, mx.y, mx.z, mx.w}, ns[4] = {mn.x, mn.y, mn.z, mn.w};
    float part = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t nx = xs[e] & ((xs[e] >> 15 & 0x00010001u) * 0xFFFFu) & 0x7FFF7FFFu;  // |kmax| where kmax < 0
      const uint32_t pn = ns[e] & ~((ns[e] >> 15 & 0x00010001u) * 0xFFFFu);              // kmin where kmin > 0
      part += (bf16_lo(nx) + bf16_hi(nx)) + (bf16_lo(pn) + bf16_hi(pn));
    }
    const unsigned grp = (chunks == 16 ? 0xFFFFu : 0xFFu) << (threadIdx.x & 31 & ~(chunks - 1));
    for (int off = chunks >> 1; off > 0; off >>= 1) part += __shfl_xor_sync(grp, part, off, chunks);
    // fp32 sums of at most 4 * D non-negative terms lose less than 2^-15 of the
    // total: scaling by (1 + 2^-14) leaves an upper bound
    if (c == 0) wsum[static_cast<int64_t>(s) * Nb_max + b] = part * (1.0f + 0x1p-14f);
  }
}

}  // namespace

cudaError_t launch_build_summary(const uint16_t *k, int64_t seg_stride, int64_t blk_stride, int64_t tok_stride,
                                 int B, int Hkv, int D, const int32_t *seq_len, int blk_begin, int blk_count,
                                 uint16_t *kmin, uint16_t *kmax, float *wsum, int Nb_max, int32_t *status,
                                 cudaStream_t st) {
  const int S = B * Hkv;
  const int64_t items = static_cast<int64_t>(S) * blk_count * (D / 8);
  const int threads = 256;
  const int64_t grid = (items + threads - 1) / threads;
  if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
  LaunchCfg lc(dim3(static_cast<unsigned>(grid)), dim3(threads), 0, st);
  return cudaLaunchKernelEx(&lc.cfg, k_build_summary, k, seg_stride, blk_stride, tok_stride, Hkv, D, seq_len,
                            blk_begin, blk_count, S, kmin, kmax, wsum, Nb_max, status);
}

}  // namespace oasis
