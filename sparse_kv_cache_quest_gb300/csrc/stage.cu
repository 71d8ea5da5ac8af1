// KV transfer: planned block tiles, host tier -> HBM slots.
//
// OasisKV paper review (xllm-io), §3 Fig. 5 ("KV Transfer Worker, CPU->GPU")
// and decode flow (the transfer plan is executed asynchronously); §5:
// background workers on their own CUDA streams, ordered with CUDA events.
//
// The host copy of the full cache is pinned, mapped host memory that the GPU
// reads directly (zero-copy): on a Grace-Blackwell node the loads travel over
// NVLink-C2C, elsewhere over PCIe.  The copy is bound by that link, not by the
// SMs, so the kernel is kept small: kCtas CTAs of 4 warps that walk the plan
// entries (segment-major) with a stride, one tile per warp at a time, all of
// the tile's 16-byte loads issued before its stores.  That keeps about a
// megabyte in flight, several times what the link needs to stay busy, in CTAs
// of about 10k registers.
//
// Placement: a staging CTA holds some two thousand host loads outstanding in
// its SM's load path for tens of microseconds, and on an SM that also runs two
// CTAs of the head-split attention (whose warps are chains of dependent shared
// memory loads and MMAs) it slows them.  The launch therefore reserves
// kReserveSmem of shared memory that the kernel does not use: the block
// scheduler then places a staging CTA only on an SM with room beside at most
// one CTA of the streaming kernels (two 84 KB attention or 102 KB scoring CTAs
// leave less than that).  Measured on the 235B-shaped decode step: 99.7 / 100.4
// -> 96.9 / 97.1 us per layer-step; no change on the 4-head layers, whose 73 KB
// attention CTAs still leave room.

#include <algorithm>

#include "common.cuh"

namespace oasis {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kCtas = 32;
constexpr int kMaxPerLane = 16;  // 16-byte loads per lane for one tile at D = 128
constexpr size_t kReserveSmem = 60 * 1024;  // shared memory reserved, not used (placement, above)

__global__ void __launch_bounds__(kThreads) k_stage(const unsigned char *__restrict__ host, int64_t seg_stride,
                                                    int host_nb, const oasis_xfer_t *__restrict__ plan,
                                                    const int32_t *__restrict__ plan_count, int cap, int S, int D,
                                                    uint16_t *__restrict__ pool, int slots, int32_t *status) {
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * kWarps;
  const int n16 = 4 * D;  // 16-byte words per tile (64*D bytes)
  const int64_t entries = static_cast<int64_t>(S) * cap;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); e < entries; e += nw) {
    const int s = static_cast<int>(e / cap), i = static_cast<int>(e % cap);
    int cnt = plan_count[s];
    if (cnt < 0 || cnt > cap) {
      if (lane == 0 && i == 0) report(status, OASIS_STATUS_PLAN_RANGE);
      cnt = cnt < 0 ? 0 : cap;
    }
    if (i >= cnt) continue;  // warp-uniform
    const oasis_xfer_t x = plan[e];
    if (x.src_block < 0 || x.src_block >= host_nb || x.dst_slot < 0 || x.dst_slot >= slots) {
      if (lane == 0) report(status, OASIS_STATUS_PLAN_RANGE);
      continue;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(host + s * seg_stride + x.src_block * (64LL * D));
    uint4 *dst = reinterpret_cast<uint4 *>(pool + (static_cast<int64_t>(s) * slots + x.dst_slot) * 32 * D);
    uint4 v[kMaxPerLane];
#pragma unroll
    for (int u = 0; u < kMaxPerLane; ++u)
      if (u * 32 + lane < n16) v[u] = src[u * 32 + lane];
#pragma unroll
    for (int u = 0; u < kMaxPerLane; ++u)
      if (u * 32 + lane < n16) dst[u * 32 + lane] = v[u];
  }
}

}  // namespace

cudaError_t launch_stage_blocks(const void *host_kv, int64_t host_seg_stride_bytes, int host_nb,
                                const oasis_xfer_t *plan, const int32_t *plan_count, int cap, int B, int Hkv,
                                int D, uint16_t *pool, int slots_per_seg, int32_t *status, cudaStream_t st) {
  if (cap == 0) return cudaSuccess;
  const int S = B * Hkv;
  const int64_t warps_needed = static_cast<int64_t>(S) * cap;
  const int grid = static_cast<int>(std::min<int64_t>(kCtas, (warps_needed + kWarps - 1) / kWarps));
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(k_stage), kReserveSmem);
  if (e != cudaSuccess) return e;
  LaunchCfg lc(dim3(grid), dim3(kThreads), kReserveSmem, st);
  return cudaLaunchKernelEx(&lc.cfg, k_stage, static_cast<const unsigned char *>(host_kv), host_seg_stride_bytes,
                            host_nb, plan, plan_count, cap, S, D, pool, slots_per_seg, status);
}

}  // namespace oasis
