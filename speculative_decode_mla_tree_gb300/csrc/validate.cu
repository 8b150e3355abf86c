// Validate mode: one verify call computed by both attention kernels, the
// tensor-core result returned, the difference measured on the device.
//
// "Deploying a Custom sm_120 Verify Kernel into Production: The Validate
// Gate", section "The Validate Mode": the custom kernel runs beside the
// reference path on the same tensors and the difference is reported before
// the custom result is trusted. Here the two paths are this library's
// tensor-core and warp-shuffle kernels.
#include <math.h>

#include "../../include/mla_tree.h"
#include "mt_common.cuh"
#include "mt_internal.h"

namespace mt {

// max |a - b| over bf16 pairs and the largest relative LSE difference; each
// warp folds its maxima into diff[] (non-negative floats order like their bits)
__global__ void __launch_bounds__(256) validate_compare_kernel(
    const uint32_t* __restrict__ a, const uint32_t* __restrict__ b, int64_t pairs,
    const float* __restrict__ la, const float* __restrict__ lb, int64_t rows, float tol,
    float* diff, int32_t* status) {
  float mo = 0.f, ml = 0.f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < pairs; i += stride) {
    const uint32_t x = a[i], y = b[i];
    const float d0 = fabsf(bf16_lo(x) - bf16_lo(y)), d1 = fabsf(bf16_hi(x) - bf16_hi(y));
    mo = fmaxf(mo, isnan(d0) ? INFINITY : d0);
    mo = fmaxf(mo, isnan(d1) ? INFINITY : d1);
  }
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < rows; i += stride) {
    const float x = la[i], y = lb[i];
    float d;
    if (isinf(x) && isinf(y) && x < 0.f && y < 0.f) d = 0.f;
    else if (isinf(x) || isinf(y) || isnan(x) || isnan(y)) d = INFINITY;
    else d = fabsf(x - y) / fmaxf(1.f, fabsf(x));
    ml = fmaxf(ml, d);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mo = fmaxf(mo, __shfl_xor_sync(0xffffffffu, mo, o));
    ml = fmaxf(ml, __shfl_xor_sync(0xffffffffu, ml, o));
  }
  if ((threadIdx.x & 31) == 0) {
    atomicMax(reinterpret_cast<int*>(diff), __float_as_int(mo));
    atomicMax(reinterpret_cast<int*>(diff) + 1, __float_as_int(ml));
    if (mo > tol || ml > tol) flag(status, MT_DEV_MISMATCH);
  }
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace mt

using namespace mt;

extern "C" {

size_t mla_tree_verify_validate_workspace_bytes(int batch, int total_q, int heads, int max_splits) {
  const size_t vb = mla_tree_verify_workspace_bytes(batch, total_q, heads, max_splits);
  if (vb == 0 || total_q < 0 || heads <= 0) return 0;
  const size_t rows = (size_t)total_q * (size_t)heads;
  return align256(vb) + align256(rows * MT_D_V * 2) + align256(rows * 4);
}

int mla_tree_verify_validate(const mt_bf16* q, const mt_bf16* kv_buf, int64_t num_slots,
                             const int32_t* kv_indices, int64_t kv_indices_len,
                             const int32_t* kv_indptr, const int32_t* qo_indptr,
                             const uint8_t* packed_mask, int64_t mask_len,
                             const int64_t* mask_indptr, int batch, int total_q, int heads,
                             float sm_scale, mt_bf16* out, float* lse, void* workspace,
                             size_t workspace_bytes, int max_splits, float tolerance, float* diff,
                             int32_t* dev_status, mt_stream_t stream) {
  if (!(tolerance >= 0.f) || !diff) return MT_EINVAL;
  if (batch < 0 || total_q < 0 || heads <= 0 || max_splits < 0 || max_splits > MT_MAX_SPLITS)
    return MT_EINVAL;
  if (batch == 0 || total_q == 0) return MT_OK;
  const size_t vb = mla_tree_verify_workspace_bytes(batch, total_q, heads, max_splits);
  const size_t need = mla_tree_verify_validate_workspace_bytes(batch, total_q, heads, max_splits);
  if (vb == 0 || need == 0) return MT_EINVAL;
  if (!workspace || (uintptr_t)workspace % 256 || workspace_bytes < need) return MT_EWORKSPACE;
  const size_t rows = (size_t)total_q * (size_t)heads;
  char* ws = static_cast<char*>(workspace);
  mt_bf16* out2 = reinterpret_cast<mt_bf16*>(ws + align256(vb));
  float* lse2 = reinterpret_cast<float*>(ws + align256(vb) + align256(rows * MT_D_V * 2));
  int rc = mla_tree_verify(q, kv_buf, num_slots, kv_indices, kv_indices_len, kv_indptr, qo_indptr,
                           packed_mask, mask_len, mask_indptr, batch, total_q, heads, sm_scale, out,
                           lse, workspace, vb, max_splits, 2, dev_status, stream);
  if (rc != MT_OK) return rc;
  rc = mla_tree_verify(q, kv_buf, num_slots, kv_indices, kv_indices_len, kv_indptr, qo_indptr,
                       packed_mask, mask_len, mask_indptr, batch, total_q, heads, sm_scale, out2,
                       lse2, workspace, vb, max_splits, 1, dev_status, stream);
  if (rc != MT_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(diff, 0, 2 * sizeof(float), s) != cudaSuccess) return MT_ECUDA;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MT_ECUDA;
  const int64_t pairs = (int64_t)rows * (MT_D_V / 2);
  int64_t blocks = (pairs + 255) / 256;
  if (blocks > (int64_t)nsm * 8) blocks = (int64_t)nsm * 8;
  if (blocks < 1) blocks = 1;
  validate_compare_kernel<<<(unsigned)blocks, 256, 0, s>>>(
      reinterpret_cast<const uint32_t*>(out), reinterpret_cast<const uint32_t*>(out2), pairs, lse,
      lse2, (int64_t)rows, tolerance, diff, dev_status);
  return cudaGetLastError() == cudaSuccess ? MT_OK : MT_ECUDA;
}

}  // extern "C"
