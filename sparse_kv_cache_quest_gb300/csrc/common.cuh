// Internal helpers shared by the kernels of liboasis.so (not part of the ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "oasis.h"

namespace oasis {

constexpr int kBlockTokens = 16;  // tokens per logical KV block

// bf16 -> fp32 widening of the low / high half of a 32-bit word (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max with NaN propagation (either input NaN -> NaN), as the IEEE maximum the
// oracle's np.maximum follows; equal to fmaxf on numbers.
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ void report(int32_t *status, int bits) {
  if (status != nullptr && bits != 0) atomicOr(status, bits);
}

// Valid tokens of sequence b, clamped to [0, max_tokens]; out-of-range lengths
// are reported once per call site through the status word.
__device__ __forceinline__ int load_len(const int32_t *seq_len, int b, int max_tokens, int32_t *status,
                                        bool reporter) {
  int L = seq_len[b];
  if (L < 0 || L > max_tokens) {
    if (reporter) report(status, OASIS_STATUS_SEQ_LEN);
    L = L < 0 ? 0 : max_tokens;
  }
  return L;
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ---- packed fp32 pairs (Blackwell f32x2 arithmetic) ------------------------
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(unsigned long long r, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
// d = a * b + c on both halves, round-to-nearest, no flush to zero.
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// ---- mbarrier / bulk-copy primitives (inline PTX, sm_90+) -------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
// One 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}" : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for phase `parity` of `bar`: false after `max_tries` failed
// polls (each try_wait itself blocks for a hardware-chosen interval).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t max_tries) {
  for (uint32_t i = 0; i < max_tries; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

}  // namespace oasis

// Launch configuration carrying the priority of the launch stream as a launch
// attribute, so that a stream capture records it in the graph's kernel node
// (a priority set only on the capturing stream does not reach the graph).
// Use in place: cfg.attrs points into this object.
namespace oasis {
struct LaunchCfg {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  LaunchCfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st) {
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    int prio = 0;
    if (cudaStreamGetPriority(st, &prio) != cudaSuccess) {
      prio = 0;
      (void)cudaGetLastError();
    }
    attr[0].id = cudaLaunchAttributePriority;
    attr[0].val.priority = prio;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  LaunchCfg(const LaunchCfg &) = delete;
  LaunchCfg &operator=(const LaunchCfg &) = delete;
  void add(const cudaLaunchAttribute &a) { attr[cfg.numAttrs++] = a; }
};
}  // namespace oasis

// Launchers implemented by the kernel translation units (host side).
namespace oasis {
cudaError_t raise_smem_limit(const void *fn, size_t smem);
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
cudaError_t launch_geometry(const void *fn, int threads, size_t smem, int *sms, int *per_sm);
cudaError_t launch_build_summary(const uint16_t *k, int64_t seg_stride, int64_t blk_stride, int64_t tok_stride,
                                 int B, int Hkv, int D, const int32_t *seq_len, int blk_begin, int blk_count,
                                 uint16_t *kmin, uint16_t *kmax, float *wsum, int Nb_max, int32_t *status,
                                 cudaStream_t st);
cudaError_t launch_score_blocks(const uint16_t *kmin, const uint16_t *kmax, int Nb_max, const uint16_t *qdraft,
                                int B, int Hkv, int G, int Nd, int D, const int32_t *seq_len, int W,
                                float *scores, int32_t *status, cudaStream_t st);
cudaError_t launch_score_blocks_tc(const uint16_t *kmin, const uint16_t *kmax, const float *wsum, int Nb_max,
                                   const uint16_t *qdraft, int B, int Hkv, int G, int Nd, int D,
                                   const int32_t *seq_len, int W, float *scores, float *radius, int32_t *status,
                                   cudaStream_t st);
cudaError_t launch_select_topk_capped(const float *scores, int Nb_max, const int32_t *seq_len, int B, int Hkv,
                                      int K, int W, int cap, const int32_t *table_in, int32_t *table_out,
                                      oasis_xfer_t *plan, int32_t *plan_count, int32_t *status, cudaStream_t st);
size_t select_tc_smem_bytes(int Nb_max, int K, int W, int cap, int D, int Nq);
cudaError_t launch_select_topk_capped_tc(float *scores, const float *radius, const uint16_t *kmin,
                                         const uint16_t *kmax, const uint16_t *qdraft, int G, int Nd, int D,
                                         int Nb_max, const int32_t *seq_len, int B, int Hkv, int K, int W, int cap,
                                         const int32_t *table_in, int32_t *table_out, oasis_xfer_t *plan,
                                         int32_t *plan_count, int32_t *status, cudaStream_t st);
cudaError_t launch_stage_blocks(const void *host_kv, int64_t host_seg_stride_bytes, int host_nb,
                                const oasis_xfer_t *plan, const int32_t *plan_count, int cap, int B, int Hkv,
                                int D, uint16_t *pool, int slots_per_seg, int32_t *status, cudaStream_t st);
cudaError_t launch_sparse_decode_attn(const uint16_t *q, const uint16_t *pool, const int32_t *table,
                                      int slots_per_seg, const int32_t *seq_len, int B, int Hkv, int G, int D,
                                      float scale, float *out, float *lse, int32_t *status, cudaStream_t st);
bool attn_tc_supports(int G, int D);
cudaError_t launch_attn_tc(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots,
                           const int32_t *seq_len, int B, int Hkv, int G, int D, float scale, float *out, float *lse,
                           int32_t *status, cudaStream_t st);
size_t attn_workspace_bytes(int B, int Hkv, int G, int D, int slots_per_seg);
size_t noalloc_scratch_bytes();
cudaError_t launch_sparse_decode_attn_noalloc(const uint16_t *q, const uint16_t *pool, const int32_t *table,
                                              int slots_per_seg, const int32_t *seq_len, int B, int Hkv, int G,
                                              int D, float scale, float *out, float *lse, int32_t *status,
                                              cudaStream_t st);
cudaError_t launch_sparse_decode_attn_ws(const uint16_t *q, const uint16_t *pool, const int32_t *table,
                                         int slots_per_seg, const int32_t *seq_len, int B, int Hkv, int G, int D,
                                         float scale, float *out, float *lse, void *ws, int32_t *status,
                                         cudaStream_t st);
}  // namespace oasis
