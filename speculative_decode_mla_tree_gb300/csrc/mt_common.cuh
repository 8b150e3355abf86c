// Device-side helpers shared by the library's kernels (never by the oracle).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/mla_tree.h"

namespace mt {

constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kRowVec = kDqk * 2 / 16;   // 72 sixteen-byte vectors per pool row
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void flag(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Request owning flattened token t: the b with qo_indptr[b] <= t < qo_indptr[b+1].
__device__ __forceinline__ int find_request(const int32_t* qo_indptr, int batch, int64_t t) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (qo_indptr[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Per-request geometry read from the device indptrs, with the consistency
// checks every attention kernel applies before touching a request's data.
struct ReqGeom {
  int64_t kv0;     // first entry of the request in kv_indices
  int L;           // key positions
  int n;           // draft rows
  int64_t q0;      // first token
  int64_t mask0;   // first mask element (byte, or word of the bit form)
  int mask_row;    // mask elements per draft row: L (bytes) or ceil(L / 32) (words)
  bool ok;
};

// mask_bits: the mask is in the bit form (rows of ceil(L / 32) uint32 words).
__device__ __forceinline__ ReqGeom request_geom(const int32_t* kv_indptr, const int32_t* qo_indptr,
                                                const int64_t* mask_indptr, int b,
                                                int64_t kv_len, int64_t mask_len, int total_q,
                                                bool mask_bits = false) {
  ReqGeom g;
  g.kv0 = kv_indptr[b];
  int64_t kv1 = kv_indptr[b + 1];
  g.q0 = qo_indptr[b];
  int64_t q1 = qo_indptr[b + 1];
  g.mask0 = mask_indptr[b];
  g.L = (int)(kv1 - g.kv0);
  g.n = (int)(q1 - g.q0);
  g.mask_row = mask_bits ? (g.L + 31) >> 5 : g.L;
  g.ok = g.kv0 >= 0 && kv1 >= g.kv0 && kv1 <= kv_len && g.q0 >= 0 && q1 >= g.q0 &&
         q1 <= total_q && g.mask0 >= 0 && g.n <= g.L &&
         g.mask0 + (int64_t)g.n * g.mask_row <= mask_len;
  return g;
}

}  // namespace mt
