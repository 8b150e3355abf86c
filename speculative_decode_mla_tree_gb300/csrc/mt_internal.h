// Host-side declarations shared by the library's translation units.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mt {

// Arguments of one verify call, passed by value to the attention kernels.
struct VerifyArgs {
  const uint16_t* q;            // bf16 [total_q, heads, 576]
  const uint16_t* kv;           // bf16 [num_slots, 576]
  int64_t num_slots;
  const int32_t* kv_indices;
  int64_t kv_len;
  const int32_t* kv_indptr;
  const int32_t* qo_indptr;
  const uint8_t* mask;           // byte mask, or nullptr when mask_bits is set
  const uint32_t* mask_bits;     // bit-form mask (rows of ceil(L / 32) words)
  int bits_mask;                 // 1: the mask is mask_bits, 0: it is mask (bytes)
  int skip_prefix;               // 1: prefix columns (j < L - n) are visible and their
                                 //   mask entries are not read
  int64_t mask_len;              // elements of that mask
  const int64_t* mask_indptr;
  int batch, total_q, heads;
  float sm_scale;
  uint16_t* out;                // bf16 [total_q, heads, 512]
  float* lse;                   // fp32 [total_q, heads]
  int max_splits;               // capacity of the partial buffers
  int32_t* status;
  // workspace views
  int32_t* ws_tok;              // [total_q] split count of each token's request (0: not
                                //   merged: unsplit, empty or inconsistent request)
  float* ws_lse;                // [max_splits][total_q*heads]
  float* ws_o;                  // [max_splits][total_q*heads][512]
};

struct WorkspaceLayout {
  size_t tok_off, lse_off, o_off, total;
};

WorkspaceLayout workspace_layout(int batch, int total_q, int heads, int max_splits);
int auto_max_splits(int batch, int total_q, int heads, int num_sms);

cudaError_t launch_draft_kv_scatter(const uint16_t* src, int64_t src_stride, const int32_t* loc,
                                    int total_q, uint16_t* kv, int64_t num_slots, int32_t* status,
                                    int num_sms, cudaStream_t stream);
cudaError_t launch_kv_indices_build(const int32_t* pidx, int64_t pidx_len, const int32_t* pptr,
                                    const int32_t* loc,
                                    const int32_t* qptr, int batch, int total_q,
                                    int32_t* kv_indices, int64_t capacity, int32_t* kv_indptr,
                                    int32_t* status, int num_sms, cudaStream_t stream);
cudaError_t launch_tree_mask_pack(const int32_t* parents, const int32_t* qptr, const int32_t* kptr,
                                  int batch, int total_q, int64_t* mask_indptr, uint8_t* mask,
                                  int64_t capacity, int32_t* status, int num_sms,
                                  cudaStream_t stream);

cudaError_t launch_tree_mask_pack_bits(const int32_t* parents, const int32_t* qptr,
                                       const int32_t* kptr, int batch, int total_q,
                                       int64_t* word_indptr, uint32_t* words, int64_t capacity,
                                       int32_t* status, int num_sms, cudaStream_t stream);

// The three marshaling steps in one launch (16-byte aligned draft rows only).
cudaError_t launch_prepare(const uint16_t* src, int64_t src_stride, const int32_t* loc,
                           const int32_t* pidx, int64_t pidx_len, const int32_t* pptr,
                           const int32_t* qptr, const int32_t* parents, int batch, int total_q,
                           uint16_t* kv, int64_t num_slots, int32_t* kv_indices, int64_t kv_capacity,
                           int32_t* kv_indptr, int64_t* word_indptr, uint32_t* words,
                           int64_t word_capacity, int32_t* status, int num_sms, cudaStream_t stream);

cudaError_t launch_verify_simt(const VerifyArgs& a, int num_sms, cudaStream_t stream);
// Whether a warp-shuffle call may split a request, i.e. needs the merge.
bool simt_may_split(int max_splits, int64_t kv_len);
cudaError_t launch_lse_merge(const VerifyArgs& a, cudaStream_t stream);
// Tensor-core path; returns cudaErrorNotSupported when it cannot serve `a`.
cudaError_t launch_verify_tc(const VerifyArgs& a, int num_sms, cudaStream_t stream);
// Kernels one tensor-core verify call launches (0 when that path cannot serve it).
int verify_tc_launches(int batch, int total_q, int heads, int max_splits);
// Test hooks of the tensor-core kernel's bounded waits (process-wide; see
// mla_tree_test_wait_limits in the public header).
void set_tc_test_hooks(int drop_item, unsigned long long limit_ns);

}  // namespace mt
