// Boundary kernels of the verify step: draft-KV scatter, KV index
// marshaling and tree-mask packing. Integer / byte work only: HBM-write
// bound, results bit-exact.
//
// "The Moment of Truth: Flipping the Switch on a Custom CUDA Verify Kernel",
// section "The Long Road to Parity": draft KV is written to out_cache_loc
// and the index array is prefix slots followed by draft slots, with the mask
// row stride prefix + draft. "The Pivot to Live Cutover", section "The
// Technical Investigation": flat mask with per-sequence offsets.
#include "mt_common.cuh"
#include "mt_internal.h"

namespace mt {

// ---------------------------------------------------------------- scatter

// One thread per 16-byte vector of a 1152-byte row: a warp moves 512
// contiguous bytes of one source row into one pool row. Block bid of nb
// blocks of 256 threads.
__device__ __forceinline__ void scatter_vec_body(const uint4* __restrict__ src, int64_t src_stride_vec,
                                                 const int32_t* __restrict__ loc, int total_q,
                                                 uint4* __restrict__ kv, int64_t num_slots,
                                                 int32_t* status, int64_t bid, int64_t nb) {
  const int64_t total = (int64_t)total_q * kRowVec;
  for (int64_t idx = bid * 256 + threadIdx.x; idx < total; idx += nb * 256) {
    const int64_t t = idx / kRowVec;
    const int v = (int)(idx - t * kRowVec);
    const int32_t slot = loc[t];
    if (slot < 0 || slot >= num_slots) {
      if (v == 0) flag(status, MT_DEV_BAD_SLOT);
      continue;
    }
    kv[(int64_t)slot * kRowVec + v] = src[t * src_stride_vec + v];
  }
}

__global__ void __launch_bounds__(256) draft_kv_scatter_vec(const uint4* __restrict__ src,
                                                            int64_t src_stride_vec,
                                                            const int32_t* __restrict__ loc,
                                                            int total_q, uint4* __restrict__ kv,
                                                            int64_t num_slots, int32_t* status) {
  scatter_vec_body(src, src_stride_vec, loc, total_q, kv, num_slots, status, blockIdx.x, gridDim.x);
}

// Fallback for sources that are not 16-byte aligned: 2-byte copies.
__global__ void __launch_bounds__(256) draft_kv_scatter_u16(const uint16_t* __restrict__ src,
                                                            int64_t src_stride,
                                                            const int32_t* __restrict__ loc,
                                                            int total_q, uint16_t* __restrict__ kv,
                                                            int64_t num_slots, int32_t* status) {
  const int64_t total = (int64_t)total_q * kDqk;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = idx / kDqk;
    const int d = (int)(idx - t * kDqk);
    const int32_t slot = loc[t];
    if (slot < 0 || slot >= num_slots) {
      if (d == 0) flag(status, MT_DEV_BAD_SLOT);
      continue;
    }
    kv[(int64_t)slot * kDqk + d] = src[t * src_stride + d];
  }
}

cudaError_t launch_draft_kv_scatter(const uint16_t* src, int64_t src_stride, const int32_t* loc,
                                    int total_q, uint16_t* kv, int64_t num_slots, int32_t* status,
                                    int num_sms, cudaStream_t stream) {
  const bool vec = ((uintptr_t)src % 16 == 0) && ((uintptr_t)kv % 16 == 0) && (src_stride % 8 == 0);
  const int64_t work = (int64_t)total_q * (vec ? kRowVec : kDqk);
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (vec)
    draft_kv_scatter_vec<<<(unsigned)blocks, 256, 0, stream>>>(
        (const uint4*)src, src_stride / 8, loc, total_q, (uint4*)kv, num_slots, status);
  else
    draft_kv_scatter_u16<<<(unsigned)blocks, 256, 0, stream>>>(src, src_stride, loc, total_q, kv,
                                                               num_slots, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- kv indices

// Chunk c of request b (of `chunks`, 256 threads each) copies positions
// j = c*256+tid, stepping by chunks*256.
__device__ __forceinline__ void indices_body(
    const int32_t* __restrict__ pidx, int64_t pidx_len, const int32_t* __restrict__ pptr,
    const int32_t* __restrict__ loc, const int32_t* __restrict__ qptr, int batch, int total_q,
    int32_t* __restrict__ kv_indices, int64_t capacity, int32_t* __restrict__ kv_indptr,
    int32_t* status, int b, int c, int chunks) {
  const int64_t p0 = pptr[b], p1 = pptr[b + 1];
  const int64_t q0 = qptr[b], q1 = qptr[b + 1];
  const int64_t base = p0 + q0;
  const int64_t P = p1 - p0, n = q1 - q0;
  if (c == 0 && threadIdx.x == 0) {
    kv_indptr[b] = (int32_t)base;
    if (b == batch - 1) {
      kv_indptr[batch] = (int32_t)(p1 + q1);
      if (q1 != total_q) flag(status, MT_DEV_BAD_INDPTR);
    }
  }
  if (P < 0 || n < 0 || p0 < 0 || q0 < 0 || p1 > pidx_len || q1 > total_q ||
      base + P + n > capacity || base + P + n > 0x7fffffffLL) {
    if (c == 0 && threadIdx.x == 0) flag(status, MT_DEV_BAD_INDPTR);
    return;
  }
  const int64_t L = P + n;
  // Thread t of chunk c copies elements c * 256 + t + k * step. Eight of
  // them are loaded before any is stored, so eight loads are in flight at
  // once: a long prefix is otherwise a chain of one memory latency per 256 x
  // chunks elements.
  const int64_t step = (int64_t)chunks * 256;
  for (int64_t j0 = (int64_t)c * 256 + threadIdx.x; j0 < L; j0 += 8 * step) {
    int32_t v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t j = j0 + u * step;
      v[u] = j < L ? (j < P ? pidx[p0 + j] : loc[q0 + (j - P)]) : 0;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t j = j0 + u * step;
      if (j < L) kv_indices[base + j] = v[u];
    }
  }
}

// grid (chunks, batch)
__global__ void __launch_bounds__(256) kv_indices_build_kernel(
    const int32_t* __restrict__ pidx, int64_t pidx_len, const int32_t* __restrict__ pptr,
    const int32_t* __restrict__ loc, const int32_t* __restrict__ qptr, int batch, int total_q,
    int32_t* __restrict__ kv_indices, int64_t capacity, int32_t* __restrict__ kv_indptr,
    int32_t* status) {
  indices_body(pidx, pidx_len, pptr, loc, qptr, batch, total_q, kv_indices, capacity, kv_indptr,
               status, blockIdx.y, blockIdx.x, gridDim.x);
}

cudaError_t launch_kv_indices_build(const int32_t* pidx, int64_t pidx_len, const int32_t* pptr,
                                    const int32_t* loc, const int32_t* qptr, int batch, int total_q,
                                    int32_t* kv_indices, int64_t capacity, int32_t* kv_indptr,
                                    int32_t* status, int num_sms, cudaStream_t stream) {
  int chunks = (2 * num_sms + batch - 1) / batch;
  if (chunks < 1) chunks = 1;
  if (chunks > 256) chunks = 256;
  dim3 grid(chunks, batch);
  kv_indices_build_kernel<<<grid, 256, 0, stream>>>(pidx, pidx_len, pptr, loc, qptr, batch, total_q,
                                                    kv_indices, capacity, kv_indptr, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- tree mask

// Block-wide sum of v; every thread gets it. red: shared scratch of 32.
__device__ __forceinline__ long long block_sum(long long v, long long* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();  // red may still be read after a previous call
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  long long t = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
  return t;
}

// Block-wide inclusive scan of v in thread order; *total gets the sum.
__device__ __forceinline__ long long block_scan(long long v, long long* red, long long* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  __syncthreads();
  if (lane == 31) red[w] = v;
  __syncthreads();
  long long before = 0, tot = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
    if (i < w) before += red[i];
    tot += red[i];
  }
  *total = tot;
  return v + before;
}

// Where request b's mask starts: the sum over requests r < b of n_r * row_r
// (row_r: its row length in mask elements, from row_len(r)), with the
// requests loaded by all the block's threads at once; bad counts earlier
// requests with n < 0 or L < n. With write_indptr the block also writes the
// offsets of every request (indptr[r + 1] = sum over r' <= r of the valid
// n * row terms), as a block-wide scan.
template <typename RowLen>
__device__ __forceinline__ void mask_offsets(const int32_t* __restrict__ qptr, int batch, int b,
                                             RowLen row_len, bool write_indptr, int64_t* indptr,
                                             long long* base, long long* bad) {
  __shared__ long long red[32];
  long long part = 0, nbad = 0;
  for (int r = threadIdx.x; r < b; r += blockDim.x) {
    const long long n = (long long)qptr[r + 1] - qptr[r];
    long long L;
    const long long row = row_len(r, &L);
    if (n < 0 || L < n) ++nbad;
    part += n * row;
  }
  *base = block_sum(part, red);
  *bad = block_sum(nbad, red);
  if (!write_indptr) return;
  if (threadIdx.x == 0) indptr[0] = 0;
  long long carry = 0;
  for (int c0 = 0; c0 < batch; c0 += blockDim.x) {
    const int r = c0 + threadIdx.x;
    long long term = 0;
    if (r < batch) {
      const long long n = (long long)qptr[r + 1] - qptr[r];
      long long L;
      const long long row = row_len(r, &L);
      term = (n >= 0 && L >= n) ? n * row : 0;
    }
    long long tot;
    const long long incl = block_scan(term, red, &tot);
    if (r < batch) indptr[r + 1] = carry + incl;
    carry += tot;
  }
}

// grid (row groups, batch). Each CTA computes its request's mask offset by
// summing n*L over earlier requests (all threads loading at once) and stages
// the request's parents in shared memory. Each warp then takes one of the
// CTA's rows at a time: it walks the row's parent chain once into its own
// bitset and writes the row: prefix bytes 1, draft byte k = bit k. Interior
// 16-byte chunks go out as one vector store; the head and tail bytes of a
// row (which may share a 16-byte chunk with the neighbouring row) are
// written byte by byte so no byte has two writers.
constexpr int kMaskThreads = 256;

__device__ __forceinline__ uint8_t mask_byte(int64_t col, int64_t P, const uint32_t* bits) {
  if (col < P) return 1;
  const int64_t k = col - P;
  return (uint8_t)((bits[k >> 5] >> (k & 31)) & 1u);
}

__global__ void __launch_bounds__(kMaskThreads) tree_mask_pack_kernel(
    const int32_t* __restrict__ parents, const int32_t* __restrict__ qptr,
    const int32_t* __restrict__ kptr, int batch, int total_q, int64_t* __restrict__ mask_indptr,
    uint8_t* __restrict__ mask, int64_t capacity, int32_t* status) {
  __shared__ uint32_t bits[kMaskThreads / 32][MT_MAX_TREE / 32];  // one ancestor bitset per warp
  const int b = blockIdx.y;
  long long s_base, s_bad;
  mask_offsets(
      qptr, batch, b,
      [&](int r, long long* L) {
        *L = (long long)kptr[r + 1] - kptr[r];
        return *L;
      },
      b == 0 && blockIdx.x == 0, mask_indptr, &s_base, &s_bad);
  const int64_t q0 = qptr[b];
  const int64_t n = (int64_t)qptr[b + 1] - q0;
  const int64_t L = (int64_t)kptr[b + 1] - kptr[b];
  const int64_t P = L - n;
  const int64_t base = s_base;
  if (s_bad || n < 0 || P < 0 || q0 < 0 || q0 + n > total_q || base + n * L > capacity) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag(status, MT_DEV_BAD_INDPTR);
    return;
  }
  if (n > MT_MAX_TREE) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag(status, MT_DEV_TREE_TOO_BIG);
    return;
  }
  const int words = (int)((n + 31) >> 5);
  // the request's parent array, staged once (-2: out of range)
  __shared__ int16_t par_s[MT_MAX_TREE];
  constexpr int kWarpsM = kMaskThreads / 32;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if ((int64_t)blockIdx.x * kWarpsM >= n) return;  // no row of this request falls to this block
  for (int64_t k = threadIdx.x; k < n; k += blockDim.x) {
    const int32_t p = parents[q0 + k];
    par_s[k] = (int16_t)(p < -1 || p >= k ? -2 : p);
  }
  __syncthreads();
  // One row per warp at a time (rows blockIdx.x * 8 + warp, stepping by
  // 8 * gridDim.x), the row's ancestor set in the warp's own bitset, so no
  // row waits for the block.
  uint32_t* wbits = bits[wid];
  for (int64_t i = (int64_t)blockIdx.x * kWarpsM + wid; i < n; i += (int64_t)gridDim.x * kWarpsM) {
    for (int w = lane; w < words; w += 32) wbits[w] = 0u;
    __syncwarp();
    if (lane == 0) {
      // Ancestor-or-self walk; parents strictly decrease, so at most n steps.
      int64_t k = i;
      while (k >= 0) {
        wbits[k >> 5] |= 1u << (k & 31);
        const int p = par_s[k];
        if (p == -2) {
          flag(status, MT_DEV_BAD_PARENT);
          break;
        }
        k = p;
      }
    }
    __syncwarp();
    uint8_t* row = mask + base + i * L;
    const uintptr_t a = (uintptr_t)row, e = a + (uintptr_t)L;
    uintptr_t a0 = (a + 15) & ~(uintptr_t)15;
    uintptr_t a1 = e & ~(uintptr_t)15;
    if (a0 > e) a0 = e;
    if (a1 < a0) a1 = a0;
    // head and tail bytes
    const int64_t head = (int64_t)(a0 - a), tail = (int64_t)(e - a1);
    for (int64_t c = lane; c < head + tail; c += 32) {
      const int64_t col = c < head ? c : (int64_t)(a1 - a) + (c - head);
      row[col] = mask_byte(col, P, wbits);
    }
    // interior 16-byte chunks
    const int64_t chunks = (int64_t)(a1 - a0) >> 4;
    for (int64_t c = lane; c < chunks; c += 32) {
      const int64_t col0 = (int64_t)(a0 - a) + (c << 4);
      uint4 v;
      if (col0 + 16 <= P) {
        v = make_uint4(0x01010101u, 0x01010101u, 0x01010101u, 0x01010101u);
      } else {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t x = 0;
#pragma unroll
          for (int y = 0; y < 4; ++y) x |= (uint32_t)mask_byte(col0 + q * 4 + y, P, wbits) << (8 * y);
          w[q] = x;
        }
        v = make_uint4(w[0], w[1], w[2], w[3]);
      }
      *(uint4*)(row + col0) = v;
    }
    __syncwarp();
  }
}

cudaError_t launch_tree_mask_pack(const int32_t* parents, const int32_t* qptr, const int32_t* kptr,
                                  int batch, int total_q, int64_t* mask_indptr, uint8_t* mask,
                                  int64_t capacity, int32_t* status, int num_sms,
                                  cudaStream_t stream) {
  // Enough row groups to cover the largest tree for moderate batches, and
  // at least ~2 CTAs per SM overall.
  int groups = (2 * num_sms + batch - 1) / batch;
  if (groups < 1) groups = 1;
  if (groups > 64) groups = 64;
  dim3 grid(groups, batch);
  tree_mask_pack_kernel<<<grid, kMaskThreads, 0, stream>>>(parents, qptr, kptr, batch, total_q,
                                                           mask_indptr, mask, capacity, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- bit-form mask
// The same visibility, one bit per (row, column): row i of request b in
// W = ceil(L / 32) words, column j in bit j % 32 of word j / 32. Words wholly
// inside the prefix are all ones; only the few words that reach the draft
// columns read the row's ancestor set.
// Key positions of request r: from kv_indptr when given, else prefix length
// (prefix_indptr) plus draft nodes (qo_indptr), which is what kv_indptr holds.
__device__ __forceinline__ long long req_len(const int32_t* kptr, const int32_t* pptr,
                                             const int32_t* qptr, int r) {
  if (kptr) return (long long)kptr[r + 1] - kptr[r];
  return ((long long)pptr[r + 1] - pptr[r]) + ((long long)qptr[r + 1] - qptr[r]);
}

// Row group g (of `groups`, kMaskThreads threads each, one row per warp at a time) of request b.
__device__ __forceinline__ void mask_bits_body(
    const int32_t* __restrict__ parents, const int32_t* __restrict__ qptr,
    const int32_t* __restrict__ kptr, const int32_t* __restrict__ pptr, int batch, int total_q,
    int64_t* __restrict__ word_indptr, uint32_t* __restrict__ words, int64_t capacity,
    int32_t* status, int b, int g, int groups) {
  __shared__ uint32_t bits[kMaskThreads / 32][MT_MAX_TREE / 32];  // one ancestor bitset per warp
  long long s_base, s_bad;
  mask_offsets(
      qptr, batch, b,
      [&](int r, long long* L) {
        *L = req_len(kptr, pptr, qptr, r);
        return (*L + 31) >> 5;
      },
      b == 0 && g == 0, word_indptr, &s_base, &s_bad);
  const int64_t q0 = qptr[b];
  const int64_t n = (int64_t)qptr[b + 1] - q0;
  const int64_t L = req_len(kptr, pptr, qptr, b);
  const int64_t P = L - n;
  const int64_t W = (L + 31) >> 5;
  const int64_t base = s_base;
  if (s_bad || n < 0 || P < 0 || q0 < 0 || q0 + n > total_q || base + n * W > capacity) {
    if (g == 0 && threadIdx.x == 0) flag(status, MT_DEV_BAD_INDPTR);
    return;
  }
  if (n > MT_MAX_TREE) {
    if (g == 0 && threadIdx.x == 0) flag(status, MT_DEV_TREE_TOO_BIG);
    return;
  }
  const int nwords = (int)((n + 31) >> 5);
  // the request's parent array, staged once (the walks below would otherwise
  // be a chain of dependent global loads, one per tree level)
  __shared__ int16_t par_s[MT_MAX_TREE];
  constexpr int kWarpsM = kMaskThreads / 32;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if ((int64_t)g * kWarpsM >= n) return;  // no row of this request falls to this block
  for (int64_t k = threadIdx.x; k < n; k += blockDim.x) {
    const int32_t p = parents[q0 + k];
    par_s[k] = (int16_t)(p < -1 || p >= k ? -2 : p);  // -2: out of range
  }
  __syncthreads();
  // One row per warp at a time (rows g * 8 + warp, stepping by 8 * groups),
  // with the row's ancestor set in the warp's own slice of `bits`, so no
  // row waits for the block.
  uint32_t* wbits = bits[wid];
  for (int64_t i = (int64_t)g * kWarpsM + wid; i < n; i += (int64_t)groups * kWarpsM) {
    for (int w = lane; w < nwords; w += 32) wbits[w] = 0u;
    __syncwarp();
    if (lane == 0) {
      // Ancestor-or-self walk; parents strictly decrease, so at most n steps.
      int64_t k = i;
      while (k >= 0) {
        wbits[k >> 5] |= 1u << (k & 31);
        const int p = par_s[k];
        if (p == -2) {
          flag(status, MT_DEV_BAD_PARENT);
          break;
        }
        k = p;
      }
    }
    __syncwarp();
    uint32_t* row = words + base + i * W;
    for (int64_t w = lane; w < W; w += 32) {
      const int64_t c0 = w << 5;
      uint32_t v;
      if (c0 + 32 <= P) {
        v = 0xffffffffu;
      } else {
        v = 0u;
#pragma unroll 4
        for (int e = 0; e < 32; ++e) {
          const int64_t col = c0 + e;
          uint32_t on = 0;
          if (col < P) on = 1;
          else if (col < L) on = (wbits[(col - P) >> 5] >> ((col - P) & 31)) & 1u;
          v |= on << e;
        }
      }
      row[w] = v;
    }
    __syncwarp();
  }
}

// grid (row groups, batch)
__global__ void __launch_bounds__(kMaskThreads) tree_mask_pack_bits_kernel(
    const int32_t* __restrict__ parents, const int32_t* __restrict__ qptr,
    const int32_t* __restrict__ kptr, int batch, int total_q, int64_t* __restrict__ word_indptr,
    uint32_t* __restrict__ words, int64_t capacity, int32_t* status) {
  mask_bits_body(parents, qptr, kptr, nullptr, batch, total_q, word_indptr, words, capacity, status,
                 blockIdx.y, blockIdx.x, gridDim.x);
}

// ---------------------------------------------------------------- fused

// The three marshaling steps of one verify step in one launch of 256-thread
// blocks: blocks [0, ns) scatter the draft rows, the next batch * ni build
// kv_indices (chunk (k / batch) of request k % batch), the last batch * nm pack
// the bit-form mask (row group (k / batch) of request k % batch). The mask
// part takes each request's key count from prefix_indptr and qo_indptr, so
// it does not wait for the kv_indptr this launch also writes.
static_assert(kMaskThreads == 256, "one block size for every part of the fused launch");
__global__ void __launch_bounds__(256) prepare_kernel(
    const uint4* __restrict__ src, int64_t src_stride_vec, const int32_t* __restrict__ loc,
    const int32_t* __restrict__ pidx, int64_t pidx_len, const int32_t* __restrict__ pptr,
    const int32_t* __restrict__ qptr, const int32_t* __restrict__ parents, int batch, int total_q,
    uint4* __restrict__ kv, int64_t num_slots, int32_t* __restrict__ kv_indices,
    int64_t kv_capacity, int32_t* __restrict__ kv_indptr, int64_t* __restrict__ word_indptr,
    uint32_t* __restrict__ words, int64_t word_capacity, int32_t* status, int ns, int ni, int nm) {
  // the verify kernel that follows may be scheduled now; it waits for this
  // grid to complete before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int k = blockIdx.x;
  if (k < ns) {
    scatter_vec_body(src, src_stride_vec, loc, total_q, kv, num_slots, status, k, ns);
  } else if (k < ns + batch * ni) {
    const int r = k - ns;
    indices_body(pidx, pidx_len, pptr, loc, qptr, batch, total_q, kv_indices, kv_capacity, kv_indptr,
                 status, r % batch, r / batch, ni);
  } else {
    const int r = k - ns - batch * ni;
    mask_bits_body(parents, qptr, nullptr, pptr, batch, total_q, word_indptr, words, word_capacity,
                   status, r % batch, r / batch, nm);
  }
}

cudaError_t launch_prepare(const uint16_t* src, int64_t src_stride, const int32_t* loc,
                           const int32_t* pidx, int64_t pidx_len, const int32_t* pptr,
                           const int32_t* qptr, const int32_t* parents, int batch, int total_q,
                           uint16_t* kv, int64_t num_slots, int32_t* kv_indices, int64_t kv_capacity,
                           int32_t* kv_indptr, int64_t* word_indptr, uint32_t* words,
                           int64_t word_capacity, int32_t* status, int num_sms, cudaStream_t stream) {
  // same work splits as the separate launches
  int64_t ns = ((int64_t)total_q * kRowVec + 255) / 256;
  if (ns > (int64_t)num_sms * 8) ns = (int64_t)num_sms * 8;
  if (ns < 1) ns = 1;
  int ni = (2 * num_sms + batch - 1) / batch;
  if (ni < 1) ni = 1;
  if (ni > 256) ni = 256;
  int nm = (2 * num_sms + batch - 1) / batch;
  if (nm < 1) nm = 1;
  if (nm > 64) nm = 64;
  const int64_t blocks = ns + (int64_t)batch * (ni + nm);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  prepare_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      (const uint4*)src, src_stride / 8, loc, pidx, pidx_len, pptr, qptr, parents, batch, total_q,
      (uint4*)kv, num_slots, kv_indices, kv_capacity, kv_indptr, word_indptr, words, word_capacity,
      status, (int)ns, ni, nm);
  return cudaGetLastError();
}

cudaError_t launch_tree_mask_pack_bits(const int32_t* parents, const int32_t* qptr,
                                       const int32_t* kptr, int batch, int total_q,
                                       int64_t* word_indptr, uint32_t* words, int64_t capacity,
                                       int32_t* status, int num_sms, cudaStream_t stream) {
  int groups = (2 * num_sms + batch - 1) / batch;
  if (groups < 1) groups = 1;
  if (groups > 64) groups = 64;
  dim3 grid(groups, batch);
  tree_mask_pack_bits_kernel<<<grid, kMaskThreads, 0, stream>>>(parents, qptr, kptr, batch, total_q,
                                                                word_indptr, words, capacity, status);
  return cudaGetLastError();
}

}  // namespace mt
