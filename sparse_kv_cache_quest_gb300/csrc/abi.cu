// extern "C" entry points of liboasis.so: host-side argument validation, then
// one launch each.  Declared and documented in include/oasis.h.
#include <cstdint>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline bool d_ok(int D) { return D == 64 || D == 128; }
inline bool segs_ok(int B, int Hkv) {
  return B >= 1 && Hkv >= 1 && static_cast<int64_t>(B) * Hkv <= 65535;
}
inline int finish(cudaError_t e) { return e == cudaSuccess ? OASIS_OK : OASIS_ECUDA; }

}  // namespace

namespace oasis {

// SM count and resident CTAs per SM of a kernel at a given dynamic shared-memory
// size, after raising the kernel's shared-memory limit to at least that size.
// Cached per process, device, kernel, block size and shared-memory size.
// Raises a kernel's dynamic shared-memory limit to at least `smem` bytes on the
// current device; never lowers it.  The limit is a property of the function, so
// a lower value set for a small launch would make a larger launch of the same
// kernel (an earlier configuration, or a captured graph replayed later) fail.
cudaError_t raise_smem_limit(const void *fn, size_t smem) {
  struct Limit {
    const void *fn;
    int dev;
    size_t smem;
  };
  static std::mutex mu;
  static std::vector<Limit> limits;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  Limit *cur = nullptr;
  for (Limit &x : limits)
    if (x.fn == fn && x.dev == dev) cur = &x;
  if (cur != nullptr && cur->smem >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (cur != nullptr)
    cur->smem = smem;
  else
    limits.push_back(Limit{fn, dev, smem});
  return cudaSuccess;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link to
// the driver library); nullptr when the driver does not provide it.
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

cudaError_t launch_geometry(const void *fn, int threads, size_t smem, int *sms, int *per_sm) {
  struct Entry {
    const void *fn;
    int dev, threads;
    size_t smem;
    int sms, per_sm;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = raise_smem_limit(fn, smem);  // on every call: a cached geometry does not mean the limit still fits
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const Entry &x : cache)
      if (x.fn == fn && x.dev == dev && x.threads == threads && x.smem == smem) {
        *sms = x.sms;
        *per_sm = x.per_sm;
        return cudaSuccess;
      }
  }
  int n = 0, p = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&p, fn, threads, smem);
  if (e != cudaSuccess) return e;
  p = p < 1 ? 1 : p;
  std::lock_guard<std::mutex> lk(mu);
  cache.push_back(Entry{fn, dev, threads, smem, n, p});
  *sms = n;
  *per_sm = p;
  return cudaSuccess;
}

}  // namespace oasis

extern "C" {

const char *oasis_strerror(int code) {
  switch (code) {
    case OASIS_OK: return "ok";
    case OASIS_EINVAL: return "invalid argument (host-side validation failed; nothing launched)";
    case OASIS_ECUDA: return "CUDA launch failed (see cudaGetLastError)";
    case OASIS_STATUS_TABLE_RANGE: return "status: a resident block is not a candidate block";
    case OASIS_STATUS_TABLE_DUP: return "status: a block is resident in two slots";
    case OASIS_STATUS_NAN_SCORE: return "status: NaN block score";
    case OASIS_STATUS_PLAN_RANGE: return "status: transfer plan entry out of range (skipped)";
    case OASIS_STATUS_SEQ_LEN: return "status: sequence length out of range (clamped)";
    case OASIS_STATUS_TIMEOUT: return "status: a bounded device wait timed out";
    default: return "unknown code";
  }
}

int oasis_abi_version(void) { return OASIS_ABI_VERSION; }

int oasis_build_summary(const uint16_t *k, int64_t seg_stride, int64_t blk_stride, int64_t tok_stride, int B,
                        int Hkv, int D, const int32_t *seq_len, int blk_begin, int blk_count, uint16_t *kmin,
                        uint16_t *kmax, float *wsum, int Nb_max, int32_t *status, oasis_stream_t stream) {
  if (!k || !seq_len || !kmin || !kmax) return OASIS_EINVAL;
  if (!d_ok(D) || !segs_ok(B, Hkv) || Nb_max < 1) return OASIS_EINVAL;
  if (blk_begin < 0 || blk_count < 0 || static_cast<int64_t>(blk_begin) + blk_count > Nb_max) return OASIS_EINVAL;
  if (seg_stride < 0 || blk_stride < 0 || tok_stride < 0) return OASIS_EINVAL;
  if ((seg_stride | blk_stride | tok_stride) & 7) return OASIS_EINVAL;
  if (!aligned16(k) || !aligned16(kmin) || !aligned16(kmax) || !aligned4(seq_len)) return OASIS_EINVAL;
  if ((status && !aligned4(status)) || (wsum && !aligned4(wsum))) return OASIS_EINVAL;
  if (blk_count == 0) return OASIS_OK;
  return finish(oasis::launch_build_summary(k, seg_stride, blk_stride, tok_stride, B, Hkv, D, seq_len, blk_begin,
                                            blk_count, kmin, kmax, wsum, Nb_max, status, stream));
}

int oasis_score_blocks(const uint16_t *kmin, const uint16_t *kmax, int Nb_max, const uint16_t *qdraft, int B,
                       int Hkv, int G, int Nd, int D, const int32_t *seq_len, int W, float *scores,
                       int32_t *status, oasis_stream_t stream) {
  if (!kmin || !kmax || !qdraft || !seq_len || !scores) return OASIS_EINVAL;
  if (!d_ok(D) || !segs_ok(B, Hkv) || Nb_max < 1 || W < 0) return OASIS_EINVAL;
  if (G < 1 || G > 16 || Nd < 1 || G * Nd > 64) return OASIS_EINVAL;
  if (!aligned16(kmin) || !aligned16(kmax) || !aligned16(qdraft) || !aligned4(seq_len) || !aligned4(scores))
    return OASIS_EINVAL;
  if (status && !aligned4(status)) return OASIS_EINVAL;
  return finish(oasis::launch_score_blocks(kmin, kmax, Nb_max, qdraft, B, Hkv, G, Nd, D, seq_len, W, scores,
                                           status, stream));
}

int oasis_score_blocks_tc(const uint16_t *kmin, const uint16_t *kmax, const float *wsum, int Nb_max,
                          const uint16_t *qdraft, int B, int Hkv, int G, int Nd, int D, const int32_t *seq_len, int W,
                          float *scores, float *radius, int32_t *status, oasis_stream_t stream) {
  if (!kmin || !kmax || !qdraft || !seq_len || !scores || !radius) return OASIS_EINVAL;
  if (!d_ok(D) || !segs_ok(B, Hkv) || Nb_max < 1 || W < 0) return OASIS_EINVAL;
  if (G < 1 || G > 16 || Nd < 1 || G * Nd > 64) return OASIS_EINVAL;
  if (!aligned16(kmin) || !aligned16(kmax) || !aligned16(qdraft) || !aligned4(seq_len) || !aligned4(scores) ||
      !aligned4(radius))
    return OASIS_EINVAL;
  if ((status && !aligned4(status)) || (wsum && !aligned4(wsum))) return OASIS_EINVAL;
  return finish(oasis::launch_score_blocks_tc(kmin, kmax, wsum, Nb_max, qdraft, B, Hkv, G, Nd, D, seq_len, W, scores,
                                              radius, status, stream));
}

int oasis_select_topk_capped(const float *scores, int Nb_max, const int32_t *seq_len, int B, int Hkv, int K,
                             int W, int cap, const int32_t *table_in, int32_t *table_out, oasis_xfer_t *plan,
                             int32_t *plan_count, int32_t *status, oasis_stream_t stream) {
  if (!scores || !seq_len || !table_in || !table_out || !plan || !plan_count || !status) return OASIS_EINVAL;
  if (!segs_ok(B, Hkv) || K < 1 || K > 1024 || W < 0 || W > 256 || cap < 0 || cap > K) return OASIS_EINVAL;
  if (Nb_max < 1 || Nb_max > 32768) return OASIS_EINVAL;
  if (!aligned4(scores) || !aligned4(seq_len) || !aligned4(table_in) || !aligned4(table_out) ||
      !aligned4(plan) || !aligned4(plan_count) || !aligned4(status))
    return OASIS_EINVAL;
  return finish(oasis::launch_select_topk_capped(scores, Nb_max, seq_len, B, Hkv, K, W, cap, table_in, table_out,
                                                 plan, plan_count, status, stream));
}

int oasis_select_topk_capped_tc(float *scores, const float *radius, const uint16_t *kmin, const uint16_t *kmax,
                                const uint16_t *qdraft, int G, int Nd, int D, int Nb_max, const int32_t *seq_len,
                                int B, int Hkv, int K, int W, int cap, const int32_t *table_in, int32_t *table_out,
                                oasis_xfer_t *plan, int32_t *plan_count, int32_t *status, oasis_stream_t stream) {
  if (!scores || !radius || !kmin || !kmax || !qdraft || !seq_len || !table_in || !table_out || !plan ||
      !plan_count || !status)
    return OASIS_EINVAL;
  if (!segs_ok(B, Hkv) || K < 1 || K > 1024 || W < 0 || W > 256 || cap < 0 || cap > K) return OASIS_EINVAL;
  if (Nb_max < 1 || Nb_max > 16384 || !d_ok(D) || G < 1 || G > 16 || Nd < 1 || G * Nd > 64) return OASIS_EINVAL;
  if (!aligned4(scores) || !aligned4(radius) || !aligned16(kmin) || !aligned16(kmax) || !aligned16(qdraft) ||
      !aligned4(seq_len) || !aligned4(table_in) || !aligned4(table_out) || !aligned4(plan) || !aligned4(plan_count) ||
      !aligned4(status))
    return OASIS_EINVAL;
  if (oasis::select_tc_smem_bytes(Nb_max, K, W, cap, D, G * Nd) > 200 * 1024) return OASIS_EINVAL;
  return finish(oasis::launch_select_topk_capped_tc(scores, radius, kmin, kmax, qdraft, G, Nd, D, Nb_max, seq_len,
                                                    B, Hkv, K, W, cap, table_in, table_out, plan, plan_count, status,
                                                    stream));
}

int oasis_stage_blocks(const void *host_kv, int64_t host_seg_stride_bytes, int host_nb, const oasis_xfer_t *plan,
                       const int32_t *plan_count, int cap, int B, int Hkv, int D, uint16_t *pool,
                       int slots_per_seg, int32_t *status, oasis_stream_t stream) {
  if (!host_kv || !plan || !plan_count || !pool || !status) return OASIS_EINVAL;
  if (!d_ok(D) || !segs_ok(B, Hkv) || cap < 0 || host_nb < 1 || slots_per_seg < 1) return OASIS_EINVAL;
  if (host_seg_stride_bytes < 0 || (host_seg_stride_bytes & 15)) return OASIS_EINVAL;
  if (!aligned16(host_kv) || !aligned16(pool) || !aligned4(plan) || !aligned4(plan_count) || !aligned4(status))
    return OASIS_EINVAL;
  return finish(oasis::launch_stage_blocks(host_kv, host_seg_stride_bytes, host_nb, plan, plan_count, cap, B, Hkv,
                                           D, pool, slots_per_seg, status, stream));
}

int oasis_sparse_decode_attn(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots_per_seg,
                             const int32_t *seq_len, int B, int Hkv, int G, int D, float scale, float *out,
                             float *lse, int32_t *status, oasis_stream_t stream) {
  if (!q || !pool || !table || !seq_len || !out) return OASIS_EINVAL;
  if (!d_ok(D) || !segs_ok(B, Hkv) || G < 1 || G > 16 || slots_per_seg < 1 || slots_per_seg > 4096)
    return OASIS_EINVAL;
  if (static_cast<int64_t>(B) * Hkv * slots_per_seg * 32 > 0x7FFFFFFF) return OASIS_EINVAL;  // pool rows
  if (!aligned16(q) || !aligned16(pool) || !aligned4(table) || !aligned4(seq_len) || !aligned4(out))
    return OASIS_EINVAL;
  if ((lse && !aligned4(lse)) || (status && !aligned4(status))) return OASIS_EINVAL;
  return finish(oasis::launch_sparse_decode_attn(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, D, scale, out,
                                                 lse, status, stream));
}

size_t oasis_attn_workspace_bytes(int B, int Hkv, int G, int D, int slots_per_seg) {
  if (!d_ok(D) || !segs_ok(B, Hkv) || G < 1 || G > 16 || slots_per_seg < 1 || slots_per_seg > 4096) return 0;
  return oasis::attn_workspace_bytes(B, Hkv, G, D, slots_per_seg);
}

int oasis_sparse_decode_attn_ws(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots_per_seg,
                                const int32_t *seq_len, int B, int Hkv, int G, int D, float scale, float *out,
                                float *lse, void *ws, size_t ws_bytes, int32_t *status, oasis_stream_t stream) {
  if (!q || !pool || !table || !seq_len || !out || !ws) return OASIS_EINVAL;
  if (!d_ok(D) || !segs_ok(B, Hkv) || G < 1 || G > 16 || slots_per_seg < 1 || slots_per_seg > 4096)
    return OASIS_EINVAL;
  if (static_cast<int64_t>(B) * Hkv * slots_per_seg * 32 > 0x7FFFFFFF) return OASIS_EINVAL;  // pool rows
  if (!aligned16(q) || !aligned16(pool) || !aligned4(table) || !aligned4(seq_len) || !aligned4(out) ||
      !aligned16(ws))
    return OASIS_EINVAL;
  if ((lse && !aligned4(lse)) || (status && !aligned4(status))) return OASIS_EINVAL;
  if (ws_bytes < oasis::attn_workspace_bytes(B, Hkv, G, D, slots_per_seg)) return OASIS_EINVAL;
  return finish(oasis::launch_sparse_decode_attn_ws(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, D, scale,
                                                    out, lse, ws, status, stream));
}

int oasis_sparse_decode_attn_noalloc(const uint16_t *q, const uint16_t *pool, const int32_t *table,
                                     int slots_per_seg, const int32_t *seq_len, int B, int Hkv, int G, int D,
                                     float scale, float *out, float *lse, int32_t *status, oasis_stream_t stream) {
  if (!q || !pool || !table || !seq_len || !out) return OASIS_EINVAL;
  if (!d_ok(D) || !segs_ok(B, Hkv) || G < 1 || G > 16 || slots_per_seg < 1 || slots_per_seg > 4096)
    return OASIS_EINVAL;
  if (static_cast<int64_t>(B) * Hkv * slots_per_seg * 32 > 0x7FFFFFFF) return OASIS_EINVAL;  // pool rows
  if (!aligned16(q) || !aligned16(pool) || !aligned4(table) || !aligned4(seq_len) || !aligned4(out))
    return OASIS_EINVAL;
  if ((lse && !aligned4(lse)) || (status && !aligned4(status))) return OASIS_EINVAL;
  if (oasis::attn_workspace_bytes(B, Hkv, G, D, slots_per_seg) > oasis::noalloc_scratch_bytes()) return OASIS_EINVAL;
  return finish(oasis::launch_sparse_decode_attn_noalloc(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, D,
                                                         scale, out, lse, status, stream));
}

int oasis_sparse_decode_attn_tc(const uint16_t *q, const uint16_t *pool, const int32_t *table, int slots_per_seg,
                                const int32_t *seq_len, int B, int Hkv, int G, int D, float scale, float *out,
                                float *lse, int32_t *status, oasis_stream_t stream) {
  if (!q || !pool || !table || !seq_len || !out) return OASIS_EINVAL;
  if (D != 128 || !segs_ok(B, Hkv) || G < 1 || G > 16 || slots_per_seg < 1 || slots_per_seg > 4096)
    return OASIS_EINVAL;
  if (static_cast<int64_t>(B) * Hkv * slots_per_seg * 32 > 0x7FFFFFFF) return OASIS_EINVAL;  // pool rows
  if (!aligned16(q) || !aligned16(pool) || !aligned4(table) || !aligned4(seq_len) || !aligned4(out))
    return OASIS_EINVAL;
  if ((lse && !aligned4(lse)) || (status && !aligned4(status))) return OASIS_EINVAL;
  return finish(oasis::launch_attn_tc(q, pool, table, slots_per_seg, seq_len, B, Hkv, G, D, scale, out, lse, status,
                                      stream));
}

}  // extern "C"
