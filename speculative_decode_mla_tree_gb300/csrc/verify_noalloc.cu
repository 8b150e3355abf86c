// mla_tree_verify_noalloc: tree-verify attention for callers that cannot
// allocate device memory.
//
// Some embedders cannot hand the library a workspace: an inference engine
// that reserves the whole GPU up front and routes every byte through its own
// arena, a plugin loaded into a host process whose allocator it does not
// own, or a latency-critical caller that must never pay for cudaMalloc's
// implicit device synchronisation. For them this entry point keeps the
// split-KV scratch in a fixed array compiled into the library.
//
// The array is a file-scope __device__ object, so every GPU that loads the
// library holds MT_NOALLOC_SCRATCH_BYTES of it until the process exits. In
// host code its name only stands in for it, so the device address is looked
// up with cudaGetSymbolAddress, once per device, on the first call made with
// that device current; make that first call outside any stream capture. The
// scratch is shared by every call on a device and keeps the last call's
// contents: the kernels write every scratch value before reading it, so
// nothing needs clearing, but two calls that overlap on the GPU (different
// streams without ordering between them) race on it.
#include <mutex>

#include "../../include/mla_tree.h"
#include "mt_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MT_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of this device's copy of the scratch array (looked up on
// first use with the device current), or nullptr if the lookup failed.
void* scratch_address(int dev) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev]) return g_scratch_addr[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
  g_scratch_addr[dev] = p;
  return p;
}

}  // namespace

extern "C" int mla_tree_verify_noalloc(const mt_bf16* q, const mt_bf16* kv_buf, int64_t num_slots,
                                       const int32_t* kv_indices, int64_t kv_indices_len,
                                       const int32_t* kv_indptr, const int32_t* qo_indptr,
                                       const uint8_t* packed_mask, int64_t mask_len,
                                       const int64_t* mask_indptr, int batch, int total_q,
                                       int heads, float sm_scale, mt_bf16* out, float* lse,
                                       int max_splits, int path, int32_t* dev_status,
                                       mt_stream_t stream) {
  if (batch < 0 || total_q < 0 || heads <= 0 || max_splits < 0 || max_splits > MT_MAX_SPLITS)
    return MT_EINVAL;
  if (batch == 0 || total_q == 0) return MT_OK;
  const size_t need = mla_tree_verify_workspace_bytes(batch, total_q, heads, max_splits);
  if (need == 0) return MT_EINVAL;
  if (need > (size_t)MT_NOALLOC_SCRATCH_BYTES) return MT_ESCRATCH;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MT_ECUDA;
  void* scratch = scratch_address(dev);
  if (!scratch) return MT_ECUDA;
  return mla_tree_verify(q, kv_buf, num_slots, kv_indices, kv_indices_len, kv_indptr, qo_indptr,
                         packed_mask, mask_len, mask_indptr, batch, total_q, heads, sm_scale, out,
                         lse, scratch, (size_t)MT_NOALLOC_SCRATCH_BYTES, max_splits, path,
                         dev_status, stream);
}
