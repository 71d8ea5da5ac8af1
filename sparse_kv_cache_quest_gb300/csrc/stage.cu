// KV transfer: planned block tiles, host tier -> HBM slots.
//
// OasisKV paper review (xllm-io), §3 Fig. 5 ("KV Transfer Worker, CPU->GPU")
// and decode flow (the transfer plan is executed asynchronously); §5:
// background workers on their own CUDA streams, ordered with CUDA events.
//
// The host copy of the full cache is pinned, mapped host memory that the GPU
// reads directly (zero-copy): on a Grace-Blackwell node the loads travel over
// NVLink-C2C, elsewhere over PCIe.  One CTA per plan entry copies one tile
// (64*D bytes) with 16-byte loads, four in flight per thread before the
// stores, so the link sees many outstanding requests.
#include "common.cuh"

namespace oasis {
namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads) k_stage(const unsigned char *__restrict__ host, int64_t seg_stride,
                                                    int host_nb, const oasis_xfer_t *__restrict__ plan,
                                                    const int32_t *__restrict__ plan_count, int cap, int D,
                                                    uint16_t *__restrict__ pool, int slots, int32_t *status) {
  const int i = blockIdx.x, s = blockIdx.y;
  int cnt = plan_count[s];
  if (cnt < 0 || cnt > cap) {
    if (threadIdx.x == 0 && i == 0) report(status, OASIS_STATUS_PLAN_RANGE);
    cnt = cnt < 0 ? 0 : cap;
  }
  if (i >= cnt) return;
  const oasis_xfer_t e = plan[static_cast<int64_t>(s) * cap + i];
  if (e.src_block < 0 || e.src_block >= host_nb || e.dst_slot < 0 || e.dst_slot >= slots) {
    if (threadIdx.x == 0) report(status, OASIS_STATUS_PLAN_RANGE);
    return;
  }
  const int64_t tile_bytes = 64LL * D;
  const uint4 *src = reinterpret_cast<const uint4 *>(host + s * seg_stride + e.src_block * tile_bytes);
  uint4 *dst = reinterpret_cast<uint4 *>(pool + (static_cast<int64_t>(s) * slots + e.dst_slot) * 32 * D);
  const int n16 = static_cast<int>(tile_bytes / 16);
  for (int base = 0; base < n16; base += 4 * kThreads) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * kThreads + threadIdx.x;
      if (idx < n16) v[u] = src[idx];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * kThreads + threadIdx.x;
      if (idx < n16) dst[idx] = v[u];
    }
  }
}

}  // namespace

cudaError_t launch_stage_blocks(const void *host_kv, int64_t host_seg_stride_bytes, int host_nb,
                                const oasis_xfer_t *plan, const int32_t *plan_count, int cap, int B, int Hkv,
                                int D, uint16_t *pool, int slots_per_seg, int32_t *status, cudaStream_t st) {
  if (cap == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(cap), static_cast<unsigned>(B * Hkv));
  k_stage<<<grid, kThreads, 0, st>>>(static_cast<const unsigned char *>(host_kv), host_seg_stride_bytes, host_nb,
                                      plan, plan_count, cap, D, pool, slots_per_seg, status);
  return cudaGetLastError();
}

}  // namespace oasis
