// C entry points: host-side checks of host-known scalars, workspace
// carving, kernel selection. No allocation, no host synchronisation, no
// read of device memory, so every call can be captured into a CUDA graph.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/mla_tree.h"
#include "mt_internal.h"

namespace mt {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

int auto_max_splits(int batch, int total_q, int heads, int num_sms) {
  (void)batch;
  const long long rows = (long long)total_q * heads;
  if (rows <= 0) return 1;
  if (num_sms <= 0) num_sms = 148;
  // Aim at about two 128-row work items per SM when every request is split.
  long long s = (2LL * num_sms * 128 + rows - 1) / rows;
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  return (int)s;
}

// Per-token split counts, then (only when a request may be split) the
// per-split LSEs and fp32 partial outputs. With max_splits == 1 no kernel
// writes or reads a partial: every row is finished in place.
WorkspaceLayout workspace_layout(int batch, int total_q, int heads, int max_splits) {
  (void)batch;
  WorkspaceLayout w;
  const size_t rows = (size_t)total_q * (size_t)heads;
  const size_t parts = max_splits > 1 ? (size_t)max_splits : 0;
  size_t off = 0;
  w.tok_off = off;
  off = align_up(off + sizeof(int32_t) * (size_t)(total_q > 0 ? total_q : 1), 256);
  w.lse_off = off;
  off = align_up(off + sizeof(float) * parts * rows, 256);
  w.o_off = off;
  off = align_up(off + sizeof(float) * parts * rows * MT_D_V, 256);
  w.total = off;
  return w;
}

}  // namespace mt

using namespace mt;

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? MT_OK : MT_ECUDA; }

extern "C" {

int mla_tree_abi_version(void) { return 100; }

const char* mla_tree_status_string(int status) {
  switch (status) {
    case MT_OK: return "ok";
    case MT_EINVAL: return "invalid argument";
    case MT_EUNSUPPORTED: return "unsupported request";
    case MT_EWORKSPACE: return "workspace missing, misaligned or too small";
    case MT_ECUDA: return "CUDA error";
    case MT_ESCRATCH: return "request needs more scratch than the built-in no-allocation buffer";
    default: return "unknown status";
  }
}

int mla_tree_draft_kv_scatter(const mt_bf16* src, int64_t src_row_stride,
                              const int32_t* out_cache_loc, int total_q, mt_bf16* kv_buf,
                              int64_t num_slots, int32_t* dev_status, mt_stream_t stream) {
  if (total_q < 0 || num_slots < 0 || src_row_stride < MT_D_QK) return MT_EINVAL;
  if (total_q == 0) return MT_OK;
  if (!src || !out_cache_loc || !kv_buf) return MT_EINVAL;
  return cuda_status(launch_draft_kv_scatter(src, src_row_stride, out_cache_loc, total_q, kv_buf,
                                             num_slots, dev_status, sm_count(),
                                             (cudaStream_t)stream));
}

int mla_tree_kv_indices_build(const int32_t* prefix_indices, int64_t prefix_indices_len,
                              const int32_t* prefix_indptr, const int32_t* out_cache_loc,
                              const int32_t* qo_indptr, int batch, int total_q,
                              int32_t* kv_indices, int64_t kv_indices_capacity,
                              int32_t* kv_indptr, int32_t* dev_status, mt_stream_t stream) {
  if (batch < 0 || total_q < 0 || kv_indices_capacity < 0 || prefix_indices_len < 0) return MT_EINVAL;
  if (batch == 0) return MT_OK;
  if (!prefix_indptr || !qo_indptr || !kv_indptr) return MT_EINVAL;
  if (kv_indices_capacity > 0 && !kv_indices) return MT_EINVAL;
  if (prefix_indices_len > 0 && !prefix_indices) return MT_EINVAL;
  if (total_q > 0 && !out_cache_loc) return MT_EINVAL;
  if (batch > 65535) return MT_EUNSUPPORTED;
  return cuda_status(launch_kv_indices_build(prefix_indices, prefix_indices_len, prefix_indptr,
                                             out_cache_loc, qo_indptr,
                                             batch, total_q, kv_indices, kv_indices_capacity,
                                             kv_indptr, dev_status, sm_count(),
                                             (cudaStream_t)stream));
}

int tree_mask_pack(const int32_t* parents, const int32_t* qo_indptr, const int32_t* kv_indptr,
                   int batch, int total_q, int64_t* mask_indptr, uint8_t* packed_mask,
                   int64_t mask_capacity, int32_t* dev_status, mt_stream_t stream) {
  if (batch < 0 || total_q < 0 || mask_capacity < 0) return MT_EINVAL;
  if (batch == 0) return MT_OK;
  if (!qo_indptr || !kv_indptr || !mask_indptr) return MT_EINVAL;
  if (total_q > 0 && !parents) return MT_EINVAL;
  if (mask_capacity > 0 && !packed_mask) return MT_EINVAL;
  if (batch > 65535) return MT_EUNSUPPORTED;
  return cuda_status(launch_tree_mask_pack(parents, qo_indptr, kv_indptr, batch, total_q,
                                           mask_indptr, packed_mask, mask_capacity, dev_status,
                                           sm_count(), (cudaStream_t)stream));
}

int tree_mask_pack_bits(const int32_t* parents, const int32_t* qo_indptr, const int32_t* kv_indptr,
                        int batch, int total_q, int64_t* mask_word_indptr, uint32_t* mask_words,
                        int64_t mask_capacity_words, int32_t* dev_status, mt_stream_t stream) {
  if (batch < 0 || total_q < 0 || mask_capacity_words < 0) return MT_EINVAL;
  if (batch == 0) return MT_OK;
  if (!qo_indptr || !kv_indptr || !mask_word_indptr) return MT_EINVAL;
  if (total_q > 0 && !parents) return MT_EINVAL;
  if (mask_capacity_words > 0 && !mask_words) return MT_EINVAL;
  if (batch > 65535) return MT_EUNSUPPORTED;
  return cuda_status(launch_tree_mask_pack_bits(parents, qo_indptr, kv_indptr, batch, total_q,
                                                mask_word_indptr, mask_words, mask_capacity_words,
                                                dev_status, sm_count(), (cudaStream_t)stream));
}

int mla_tree_prepare(const mt_bf16* draft_kv, int64_t draft_row_stride,
                     const int32_t* out_cache_loc, const int32_t* prefix_indices,
                     int64_t prefix_indices_len, const int32_t* prefix_indptr,
                     const int32_t* qo_indptr, const int32_t* parents, int batch, int total_q,
                     mt_bf16* kv_buf, int64_t num_slots, int32_t* kv_indices,
                     int64_t kv_indices_capacity, int32_t* kv_indptr, int64_t* mask_word_indptr,
                     uint32_t* mask_words, int64_t mask_capacity_words, int32_t* dev_status,
                     mt_stream_t stream) {
  if (batch < 0 || total_q < 0 || num_slots < 0 || kv_indices_capacity < 0 ||
      prefix_indices_len < 0 || mask_capacity_words < 0 || draft_row_stride < MT_D_QK)
    return MT_EINVAL;
  if (batch == 0) return MT_OK;
  if (!prefix_indptr || !qo_indptr || !kv_indptr || !mask_word_indptr || !kv_buf) return MT_EINVAL;
  if (total_q > 0 && (!draft_kv || !out_cache_loc || !parents)) return MT_EINVAL;
  if (kv_indices_capacity > 0 && !kv_indices) return MT_EINVAL;
  if (prefix_indices_len > 0 && !prefix_indices) return MT_EINVAL;
  if (mask_capacity_words > 0 && !mask_words) return MT_EINVAL;
  if ((uintptr_t)draft_kv % 16 || (uintptr_t)kv_buf % 16 || draft_row_stride % 8) return MT_EINVAL;
  if (batch > 65535) return MT_EUNSUPPORTED;
  return cuda_status(launch_prepare(draft_kv, draft_row_stride, out_cache_loc, prefix_indices,
                                    prefix_indices_len, prefix_indptr, qo_indptr, parents, batch,
                                    total_q, kv_buf, num_slots, kv_indices, kv_indices_capacity,
                                    kv_indptr, mask_word_indptr, mask_words, mask_capacity_words,
                                    dev_status, sm_count(), (cudaStream_t)stream));
}

size_t mla_tree_verify_workspace_bytes(int batch, int total_q, int heads, int max_splits) {
  if (batch < 0 || total_q < 0 || heads < 0 || max_splits < 0 || max_splits > MT_MAX_SPLITS) return 0;
  if (max_splits == 0) max_splits = auto_max_splits(batch, total_q, heads, sm_count());
  return workspace_layout(batch, total_q, heads, max_splits).total;
}

int mla_tree_test_wait_limits(int drop_item, int64_t wait_limit_ns) {
  if (drop_item < -1 || wait_limit_ns < 0) return MT_EINVAL;
  set_tc_test_hooks(drop_item, (unsigned long long)wait_limit_ns);
  return MT_OK;
}

int mla_tree_verify_launch_count(int batch, int total_q, int heads, int64_t kv_indices_len,
                                 int max_splits, int path) {
  if (batch < 0 || total_q < 0 || heads <= 0 || kv_indices_len < 0 || max_splits < 0 ||
      max_splits > MT_MAX_SPLITS || path < 0 || path > 2)
    return 0;
  if (batch == 0 || total_q == 0) return 0;
  if (max_splits == 0) max_splits = auto_max_splits(batch, total_q, heads, sm_count());
  bool use_tc = path == 2 || (path == 0 && (long long)total_q * heads >= 128LL * batch);
  if (use_tc) {
    const int n = verify_tc_launches(batch, total_q, heads, max_splits);
    if (n > 0) return n;
    if (path == 2) return 0;
  }
  return simt_may_split(max_splits, kv_indices_len) ? 2 : 1;
}

}  // extern "C"

// One verify call with either mask form: bits = 0 uses packed_mask (bytes),
// bits = 1 uses mask_words; mask_len counts the elements of that mask.
// skip_prefix = 1: prefix columns are visible without reading the mask.
static int verify_common(const mt_bf16* q, const mt_bf16* kv_buf, int64_t num_slots,
                         const int32_t* kv_indices, int64_t kv_indices_len,
                         const int32_t* kv_indptr, const int32_t* qo_indptr, int bits,
                         int skip_prefix,
                         const uint8_t* packed_mask, const uint32_t* mask_words, int64_t mask_len,
                         const int64_t* mask_indptr, int batch, int total_q, int heads,
                         float sm_scale, mt_bf16* out, float* lse, void* workspace,
                         size_t workspace_bytes, int max_splits, int path, int32_t* dev_status,
                         mt_stream_t stream) {
  if (batch < 0 || total_q < 0 || heads <= 0 || num_slots < 0 || kv_indices_len < 0 ||
      mask_len < 0 || max_splits < 0 || max_splits > MT_MAX_SPLITS || path < 0 || path > 2)
    return MT_EINVAL;
  if (!isfinite(sm_scale)) return MT_EINVAL;
  if (batch == 0 || total_q == 0) return MT_OK;
  if (!q || !kv_buf || !kv_indptr || !qo_indptr || !mask_indptr || !out || !lse) return MT_EINVAL;
  if (kv_indices_len > 0 && !kv_indices) return MT_EINVAL;
  if (mask_len > 0 && (bits ? !mask_words : !packed_mask)) return MT_EINVAL;
  if ((uintptr_t)q % 16 || (uintptr_t)kv_buf % 16 || (uintptr_t)out % 16 || (uintptr_t)lse % 4)
    return MT_EINVAL;
  if ((long long)total_q * heads > (1LL << 31) / MT_D_V) return MT_EUNSUPPORTED;
  const int nsm = sm_count();
  if (max_splits == 0) max_splits = auto_max_splits(batch, total_q, heads, nsm);
  const WorkspaceLayout wl = workspace_layout(batch, total_q, heads, max_splits);
  if (!workspace || (uintptr_t)workspace % 256 || workspace_bytes < wl.total) return MT_EWORKSPACE;

  VerifyArgs a;
  a.q = q;
  a.kv = kv_buf;
  a.num_slots = num_slots;
  a.kv_indices = kv_indices;
  a.kv_len = kv_indices_len;
  a.kv_indptr = kv_indptr;
  a.qo_indptr = qo_indptr;
  a.mask = bits ? nullptr : packed_mask;
  a.mask_bits = bits ? mask_words : nullptr;
  a.bits_mask = bits ? 1 : 0;
  a.skip_prefix = skip_prefix ? 1 : 0;
  a.mask_len = mask_len;
  a.mask_indptr = mask_indptr;
  a.batch = batch;
  a.total_q = total_q;
  a.heads = heads;
  a.sm_scale = sm_scale;
  a.out = out;
  a.lse = lse;
  a.max_splits = max_splits;
  a.status = dev_status;
  char* ws = (char*)workspace;
  a.ws_tok = (int32_t*)(ws + wl.tok_off);
  a.ws_lse = (float*)(ws + wl.lse_off);
  a.ws_o = (float*)(ws + wl.o_off);

  cudaStream_t s = (cudaStream_t)stream;
  // Automatic choice: the tensor-core kernel when a request's rows fill a
  // 128-row tile on average, else the warp-shuffle kernel.
  bool use_tc = path == 2;
  if (path == 0) use_tc = (long long)total_q * heads >= 128LL * batch;
  if (use_tc) {
    cudaError_t e = launch_verify_tc(a, nsm, s);
    if (e == cudaErrorNotSupported) {
      if (path == 2) return MT_EUNSUPPORTED;
      use_tc = false;
    } else {
      return cuda_status(e);
    }
  }
  cudaError_t e = launch_verify_simt(a, nsm, s);
  if (e != cudaSuccess) return MT_ECUDA;
  if (simt_may_split(max_splits, kv_indices_len)) e = launch_lse_merge(a, s);
  return cuda_status(e);
}

extern "C" {

int mla_tree_verify(const mt_bf16* q, const mt_bf16* kv_buf, int64_t num_slots,
                    const int32_t* kv_indices, int64_t kv_indices_len, const int32_t* kv_indptr,
                    const int32_t* qo_indptr, const uint8_t* packed_mask, int64_t mask_len,
                    const int64_t* mask_indptr, int batch, int total_q, int heads, float sm_scale,
                    mt_bf16* out, float* lse, void* workspace, size_t workspace_bytes,
                    int max_splits, int path, int32_t* dev_status, mt_stream_t stream) {
  return verify_common(q, kv_buf, num_slots, kv_indices, kv_indices_len, kv_indptr, qo_indptr, 0, 0,
                       packed_mask, nullptr, mask_len, mask_indptr, batch, total_q, heads,
                       sm_scale, out, lse, workspace, workspace_bytes, max_splits, path,
                       dev_status, stream);
}

int mla_tree_verify_bits(const mt_bf16* q, const mt_bf16* kv_buf, int64_t num_slots,
                         const int32_t* kv_indices, int64_t kv_indices_len,
                         const int32_t* kv_indptr, const int32_t* qo_indptr,
                         const uint32_t* mask_words, int64_t mask_len_words,
                         const int64_t* mask_word_indptr, int batch, int total_q, int heads,
                         float sm_scale, mt_bf16* out, float* lse, void* workspace,
                         size_t workspace_bytes, int max_splits, int path, int32_t* dev_status,
                         mt_stream_t stream) {
  return verify_common(q, kv_buf, num_slots, kv_indices, kv_indices_len, kv_indptr, qo_indptr, 1, 0,
                       nullptr, mask_words, mask_len_words,
                       mask_word_indptr, batch, total_q, heads, sm_scale, out, lse, workspace,
                       workspace_bytes, max_splits, path, dev_status, stream);
}

int mla_tree_verify_masked(const mt_bf16* q, const mt_bf16* kv_buf, int64_t num_slots,
                           const int32_t* kv_indices, int64_t kv_indices_len,
                           const int32_t* kv_indptr, const int32_t* qo_indptr, const void* mask,
                           int64_t mask_len, const int64_t* mask_indptr, int mask_flags,
                           int batch, int total_q, int heads, float sm_scale, mt_bf16* out,
                           float* lse, void* workspace, size_t workspace_bytes, int max_splits,
                           int path, int32_t* dev_status, mt_stream_t stream) {
  if (mask_flags & ~(MT_MASK_BITS | MT_MASK_SKIP_PREFIX)) return MT_EINVAL;
  const int bits = (mask_flags & MT_MASK_BITS) ? 1 : 0;
  if (bits && (uintptr_t)mask % 4) return MT_EINVAL;
  return verify_common(q, kv_buf, num_slots, kv_indices, kv_indices_len, kv_indptr, qo_indptr, bits,
                       (mask_flags & MT_MASK_SKIP_PREFIX) ? 1 : 0,
                       bits ? nullptr : (const uint8_t*)mask, bits ? (const uint32_t*)mask : nullptr,
                       mask_len, mask_indptr, batch, total_q, heads, sm_scale, out, lse, workspace,
                       workspace_bytes, max_splits, path, dev_status, stream);
}

}  // extern "C"
