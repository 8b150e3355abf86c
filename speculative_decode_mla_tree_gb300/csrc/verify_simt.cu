// Warp-shuffle (SIMT) tree-verify attention and the split-KV LSE merge.
//
// The path for small trees, where heads x draft rows cannot fill a tensor-core
// tile (the pages' live call had 9 rows x 8 heads = 72: "Flipping the
// Switch", section "The Long Road to Parity"). Split-KV flash-decode with a
// log-sum-exp merge, after "Flipping the Switch", section "The Broader
// Context".
//
// One warp owns one draft token and up to kRows heads of it, for one KV
// split. Lane l holds latent dims [16 l, 16 l + 16) and rope dims
// [512 + 2 l, 512 + 2 l + 2) of the query rows, so one pool row is read
// with two 16-byte loads and one 4-byte load per lane (1152 contiguous bytes
// per warp) and serves both the score (all 576 dims) and the value update
// (the 512 latent dims the lane already holds). Scores are reduced with xor
// shuffles, so every lane holds the same bits; the online softmax runs in
// the log2 domain with sm_scale * log2(e) folded into q.
#include <cuda_fp16.h>
#include <math.h>

#include "mt_common.cuh"
#include "mt_internal.h"

namespace mt {

constexpr int kRows = 4;          // heads per warp
constexpr int kWarps = 4;         // warps per CTA
constexpr int kMinChunk = 8;      // smallest KV split worth a warp (keys are a serial latency chain)

__device__ __forceinline__ int simt_splits(int L, int max_splits, int* chunk) {
  int c = (L + max_splits - 1) / max_splits;
  if (c < kMinChunk) c = kMinChunk;
  *chunk = c;
  const int s = (L + c - 1) / c;
  return s < 1 ? 1 : s;
}

__device__ __forceinline__ void load_row18(const uint16_t* row, int lane, float scale, float* f) {
  const uint4 x0 = __ldg(reinterpret_cast<const uint4*>(row) + 2 * lane);
  const uint4 x1 = __ldg(reinterpret_cast<const uint4*>(row) + 2 * lane + 1);
  const uint32_t rp = __ldg(reinterpret_cast<const uint32_t*>(row + kDv) + lane);
  const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    f[2 * e] = bf16_lo(w[e]) * scale;
    f[2 * e + 1] = bf16_hi(w[e]) * scale;
  }
  f[16] = bf16_lo(rp) * scale;
  f[17] = bf16_hi(rp) * scale;
}

__global__ void __launch_bounds__(kWarps * 32) verify_simt_kernel(const VerifyArgs a) {
  // launched as a programmatic dependent of the previous kernel in the
  // stream: wait for it to complete before reading anything it may write
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int hg_count = (a.heads + kRows - 1) / kRows;
  const int64_t t = wid / hg_count;
  const int h0 = (int)(wid - t * hg_count) * kRows;
  if (t >= a.total_q) return;
  const int split = blockIdx.y;
  const int b = find_request(a.qo_indptr, a.batch, t);
  const ReqGeom g = request_geom(a.kv_indptr, a.qo_indptr, a.mask_indptr, b, a.kv_len,
                                 a.mask_len, a.total_q, a.bits_mask != 0);
  if (!g.ok || t < g.q0 || t >= g.q0 + g.n) {
    if (lane == 0 && split == 0) {
      flag(a.status, MT_DEV_BAD_INDPTR);
      if (h0 == 0) a.ws_tok[t] = 0;  // nothing to merge for this token
    }
    return;
  }
  int chunk;
  const int S = simt_splits(g.L, a.max_splits, &chunk);
  if (split == 0 && lane == 0 && h0 == 0) a.ws_tok[t] = S;
  if (split >= S) return;
  const int j0 = split * chunk;
  const int j1 = min(g.L, j0 + chunk);

  const float qscale = a.sm_scale * kLog2e;
  float qv[kRows][18];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int h = h0 + r;
    if (h < a.heads) {
      load_row18(a.q + ((int64_t)t * a.heads + h) * kDqk, lane, qscale, qv[r]);
    } else {
#pragma unroll
      for (int e = 0; e < 18; ++e) qv[r][e] = 0.f;
    }
  }

  float m[kRows], l[kRows], acc[kRows][16];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[r][e] = 0.f;
  }

  // this token's mask row: L bytes, or ceil(L / 32) words of the bit form
  const int64_t mrow0 = g.mask0 + (t - g.q0) * (int64_t)g.mask_row;
  const int32_t* idx = a.kv_indices + g.kv0;
  const int pre = a.skip_prefix ? g.L - g.n : 0;  // columns visible without a mask read
  for (int j = j0; j < j1; ++j) {
    const int32_t slot = __ldg(idx + j);
    if (slot < 0 || slot >= a.num_slots) {
      if (lane == 0) flag(a.status, MT_DEV_BAD_SLOT);
      continue;
    }
    const bool vis = j < pre ? true
                     : a.bits_mask ? ((__ldg(a.mask_bits + mrow0 + (j >> 5)) >> (j & 31)) & 1u)
                                   : __ldg(a.mask + mrow0 + j) != 0;
    if (!vis) continue;
    float kf[18];
    load_row18(a.kv + (int64_t)slot * kDqk, lane, 1.f, kf);
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < 18; ++e) d = fmaf(qv[r][e], kf[e], d);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      if (d > m[r]) {
        const float c = exp2f(m[r] - d);
        l[r] *= c;
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[r][e] *= c;
        m[r] = d;
      }
      const float p = exp2f(d - m[r]);
      l[r] += p;
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[r][e] = fmaf(p, kf[e], acc[r][e]);
    }
  }

  const int64_t R = (int64_t)a.total_q * a.heads;
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int h = h0 + r;
    if (h >= a.heads) continue;
    const int64_t row = t * a.heads + h;
    const bool any = l[r] > 0.f;
    const float inv = any ? 1.f / l[r] : 0.f;
    const float row_lse = any ? (m[r] + log2f(l[r])) * kLn2 : -INFINITY;
    if (S == 1) {
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(acc[r][2 * e] * inv, acc[r][2 * e + 1] * inv);
        w[e] = *reinterpret_cast<const uint32_t*>(&v);
      }
      uint4* dst = reinterpret_cast<uint4*>(a.out + row * kDv) + 2 * lane;
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      if (lane == 0) a.lse[row] = row_lse;
    } else {
      float4* dst = reinterpret_cast<float4*>(a.ws_o + ((int64_t)split * R + row) * kDv) + 4 * lane;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        dst[e] = make_float4(acc[r][4 * e] * inv, acc[r][4 * e + 1] * inv, acc[r][4 * e + 2] * inv,
                             acc[r][4 * e + 3] * inv);
      if (lane == 0) a.ws_lse[(int64_t)split * R + row] = row_lse;
    }
  }
}

cudaError_t launch_verify_simt(const VerifyArgs& a, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  const int hg_count = (a.heads + kRows - 1) / kRows;
  const int64_t warps = (int64_t)a.total_q * hg_count;
  const int64_t blocks = (warps + kWarps - 1) / kWarps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, (unsigned)a.max_splits);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_simt_kernel, a);
}

// ---------------------------------------------------------------- merge

// lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * o_s  -> bf16.
// One CTA per (token, group of heads). Each thread owns the 16 bytes of a
// partial row that one vector load brings in: 8 dims of an fp16 partial
// (tensor-core path) or 4 of an fp32 one (warp-shuffle path). The producing
// kernel records each token's split count, so one load decides the work.
// Then the LSEs and partials of up to kMergeGroup splits are loaded at once:
// two dependent memory rounds per row. More splits are taken in further
// groups of the same size, with the running maximum rescaled between
// groups. Tokens of unsplit requests were finished in place.
constexpr int kMergeThreads = 128;
constexpr int kMergeGroup = 12;

template <typename P>
struct MergeShape {
  static constexpr int kVec = 16 / (int)sizeof(P);              // dims per thread
  static constexpr int kThreadsPerHead = kDv / kVec;
  static constexpr int kHeads = kMergeThreads / kThreadsPerHead;  // heads per CTA
};

__device__ __forceinline__ void unpack16(const uint4 u, const float*, float (&x)[4]) {
  x[0] = __uint_as_float(u.x);
  x[1] = __uint_as_float(u.y);
  x[2] = __uint_as_float(u.z);
  x[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack16(const uint4 u, const __half*, float (&x)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
    x[2 * e] = f.x;
    x[2 * e + 1] = f.y;
  }
}

template <typename P>
__global__ void __launch_bounds__(kMergeThreads) lse_merge_kernel(const VerifyArgs a) {
  using Shape = MergeShape<P>;
  constexpr int kVec = Shape::kVec;
  const int tid = threadIdx.x;
  const int hl = tid / Shape::kThreadsPerHead, dv = tid % Shape::kThreadsPerHead;
  const int64_t t = blockIdx.x;
  // When launched as a dependent grid of the producing kernel, wait for it
  // to complete (and its writes to be visible) before reading anything it
  // wrote; otherwise this returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // split count of the token's request, recorded by the producing kernel
  // (0 or 1: nothing to merge)
  const int ns = __ldcg(a.ws_tok + t);
  if (ns <= 1 || ns > a.max_splits) return;
  const int h = blockIdx.y * Shape::kHeads + hl;
  if (h >= a.heads) return;
  const int64_t R = (int64_t)a.total_q * a.heads;
  const int64_t row = t * a.heads + h;
  const P* base = reinterpret_cast<const P*>(a.ws_o) + row * kDv + kVec * dv;
  const int64_t step = R * kDv;  // elements between two splits of one row
  float acc[kVec];
#pragma unroll
  for (int e = 0; e < kVec; ++e) acc[e] = 0.f;
  float tot = 0.f, mx = -INFINITY;
#pragma unroll 1
  for (int g0 = 0; g0 < ns; g0 += kMergeGroup) {
    float ls[kMergeGroup];
    uint4 v[kMergeGroup];
    const float* pl = a.ws_lse + (int64_t)g0 * R + row;
    const P* po = base + (int64_t)g0 * step;
#pragma unroll
    for (int s = 0; s < kMergeGroup; ++s, pl += R, po += step)
      if (g0 + s < ns) {
        ls[s] = __ldg(pl);
        v[s] = __ldg(reinterpret_cast<const uint4*>(po));
      }
    float gm = -INFINITY;
#pragma unroll
    for (int s = 0; s < kMergeGroup; ++s)
      if (g0 + s < ns) gm = fmaxf(gm, ls[s]);
    if (gm == -INFINITY) continue;  // every split of this group saw nothing
    if (gm > mx) {  // rescale what earlier groups summed (nothing on the first)
      const float c = exp2f((mx - gm) * kLog2e);
      tot *= c;
#pragma unroll
      for (int e = 0; e < kVec; ++e) acc[e] *= c;
      mx = gm;
    }
#pragma unroll
    for (int s = 0; s < kMergeGroup; ++s)
      if (g0 + s < ns && ls[s] != -INFINITY) {
        const float w = exp2f((ls[s] - mx) * kLog2e);
        float x[kVec];
        unpack16(v[s], static_cast<const P*>(nullptr), x);
        tot += w;
#pragma unroll
        for (int e = 0; e < kVec; ++e) acc[e] = fmaf(w, x[e], acc[e]);
      }
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  uint32_t o[kVec / 2];
#pragma unroll
  for (int e = 0; e < kVec / 2; ++e) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv);
    o[e] = *reinterpret_cast<const uint32_t*>(&b);
  }
  uint16_t* dst = a.out + row * kDv + kVec * dv;
  if (kVec == 8)
    *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2 % (kVec / 2)], o[3 % (kVec / 2)]);  // kVec / 2 == 4 here
  else
    *reinterpret_cast<uint2*>(dst) = make_uint2(o[0], o[1]);
  if (dv == 0) a.lse[row] = tot > 0.f ? mx + logf(tot) : -INFINITY;
}

cudaError_t launch_lse_merge(const VerifyArgs& a, cudaStream_t stream) {
  // Programmatic dependent launch: the merge grid is scheduled while the
  // producing kernel drains and waits on-device for its completion, which
  // hides the launch gap between the two.
  cudaLaunchConfig_t cfg = {};
  const int heads_per_cta = a.partial_f16 ? MergeShape<__half>::kHeads : MergeShape<float>::kHeads;
  cfg.gridDim = dim3((unsigned)a.total_q, (unsigned)((a.heads + heads_per_cta - 1) / heads_per_cta));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (a.partial_f16) return cudaLaunchKernelEx(&cfg, lse_merge_kernel<__half>, a);
  return cudaLaunchKernelEx(&cfg, lse_merge_kernel<float>, a);
}

}  // namespace mt
