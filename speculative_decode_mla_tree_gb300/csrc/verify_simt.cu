// Warp-shuffle (SIMT) tree-verify attention and the split-KV LSE merge.
//
// The path for small trees, where heads x draft rows cannot fill a tensor-core
// tile (the pages' live call had 9 rows x 8 heads = 72: "Flipping the
// Switch", section "The Long Road to Parity"). Split-KV flash-decode with a
// log-sum-exp merge, after "Flipping the Switch", section "The Broader
// Context".
//
// One CTA of kWarps warps owns one draft token, up to kRows heads of it and
// one KV split. The warps cut the split's key range into kWarps contiguous
// pieces and run an online softmax over their piece; the pieces are merged
// in shared memory at the end, so a request of up to kMinKeysY keys needs
// no split and no merge launch. Lane l holds latent dims [16 l, 16 l + 16)
// and rope dims [512 + 2 l, 512 + 2 l + 2) of the query rows, so one pool
// row is read with two 16-byte loads and one 4-byte load per lane (1152
// contiguous bytes per warp) and serves both the score (all 576 dims) and
// the value update (the 512 latent dims the lane already holds). Keys go
// two at a time, so their row loads overlap. Scores are reduced with xor
// shuffles, so every lane holds the same bits; the online softmax runs in
// the log2 domain with sm_scale * log2(e) folded into q.
#include <math.h>

#include <mutex>

#include "mt_common.cuh"
#include "mt_internal.h"

namespace mt {

constexpr int kRows = 4;          // heads per CTA
constexpr int kWarps = 8;         // warps per CTA, splitting its key range
constexpr int kMinKeysY = 256;    // smallest KV split of the grid (keys)
constexpr int kSimtSmem = kWarps * kRows * kDv * 4;  // the warps' partial outputs

__device__ __forceinline__ int simt_splits(int L, int max_splits, int* chunk) {
  int c = (L + max_splits - 1) / max_splits;
  if (c < kMinKeysY) c = kMinKeysY;
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
  extern __shared__ float part_o[];             // [kWarps][kRows][512]
  __shared__ float part_m[kWarps][kRows], part_l[kWarps][kRows];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int hg_count = (a.heads + kRows - 1) / kRows;
  const int64_t t = blockIdx.x / hg_count;
  const int h0 = (int)(blockIdx.x - t * hg_count) * kRows;
  if (t >= a.total_q) return;
  const int split = blockIdx.y;
  const int b = find_request(a.qo_indptr, a.batch, t);
  const ReqGeom g = request_geom(a.kv_indptr, a.qo_indptr, a.mask_indptr, b, a.kv_len,
                                 a.mask_len, a.total_q, a.bits_mask != 0);
  if (!g.ok || t < g.q0 || t >= g.q0 + g.n) {
    if (tid == 0 && split == 0) {
      flag(a.status, MT_DEV_BAD_INDPTR);
      if (h0 == 0) a.ws_tok[t] = 0;  // nothing to merge for this token
    }
    return;
  }
  int chunk;
  const int S = simt_splits(g.L, a.max_splits, &chunk);
  if (split == 0 && tid == 0 && h0 == 0) a.ws_tok[t] = S;
  if (split >= S) return;
  const int j0 = split * chunk;
  const int j1 = min(g.L, j0 + chunk);
  const int per = (j1 - j0 + kWarps - 1) / kWarps;  // this warp's piece
  const int wj0 = min(j1, j0 + w * per), wj1 = min(j1, wj0 + per);

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
  auto visible = [&](int j) -> bool {
    return j < pre ? true
           : a.bits_mask ? ((__ldg(a.mask_bits + mrow0 + (j >> 5)) >> (j & 31)) & 1u) != 0
                         : __ldg(a.mask + mrow0 + j) != 0;
  };
  // one key of row r: its score and the online-softmax update
  auto update = [&](int r, const float (&kf)[18]) {
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
  };
  // The piece goes in batches of 32 keys: lane i reads key i's slot and
  // visibility first (one round of loads for the batch; a bad slot is
  // flagged and skipped), then the keys are taken two at a time, so the
  // only loads left in the key loop are the rows themselves.
  for (int jb = wj0; jb < wj1; jb += 32) {
    const int nb = min(32, wj1 - jb);
    int32_t my_slot = 0;
    bool my_vis = false;
    if (lane < nb) {
      my_slot = __ldg(idx + jb + lane);
      const bool ok = my_slot >= 0 && my_slot < a.num_slots;
      if (!ok) flag(a.status, MT_DEV_BAD_SLOT);
      my_vis = ok && visible(jb + lane);
    }
    const uint32_t vis = __ballot_sync(0xffffffffu, my_vis);
    for (int i = 0; i < nb; i += 2) {
      const int32_t s0 = __shfl_sync(0xffffffffu, my_slot, i);
      const int32_t s1 = __shfl_sync(0xffffffffu, my_slot, (i + 1) & 31);
      const bool v0 = (vis >> i) & 1u, v1 = i + 1 < nb && ((vis >> (i + 1)) & 1u);
      float k0[18], k1[18];
      if (v0) load_row18(a.kv + (int64_t)s0 * kDqk, lane, 1.f, k0);
      if (v1) load_row18(a.kv + (int64_t)s1 * kDqk, lane, 1.f, k1);
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        if (v0) update(r, k0);
        if (v1) update(r, k1);
      }
    }
  }

  // merge the warps' pieces
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    if (lane == 0) {
      part_m[w][r] = m[r];
      part_l[w][r] = l[r];
    }
    float4* dst = reinterpret_cast<float4*>(part_o + (w * kRows + r) * kDv + 16 * lane);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      dst[e] = make_float4(acc[r][4 * e], acc[r][4 * e + 1], acc[r][4 * e + 2], acc[r][4 * e + 3]);
  }
  __syncthreads();
  const int r = tid >> 6, d0 = (tid & 63) * 8;  // this thread's head and 8 dims
  const int h = h0 + r;
  if (h >= a.heads) return;
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < kWarps; ++k) mx = fmaxf(mx, part_m[k][r]);
  float tot = 0.f, o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = 0.f;
  if (mx != -INFINITY) {
#pragma unroll
    for (int k = 0; k < kWarps; ++k) {
      const float mk = part_m[k][r];
      if (mk == -INFINITY) continue;
      const float c = exp2f(mk - mx);
      tot = fmaf(c, part_l[k][r], tot);
      const float4* src = reinterpret_cast<const float4*>(part_o + (k * kRows + r) * kDv + d0);
      const float4 x0 = src[0], x1 = src[1];
      o[0] = fmaf(c, x0.x, o[0]); o[1] = fmaf(c, x0.y, o[1]);
      o[2] = fmaf(c, x0.z, o[2]); o[3] = fmaf(c, x0.w, o[3]);
      o[4] = fmaf(c, x1.x, o[4]); o[5] = fmaf(c, x1.y, o[5]);
      o[6] = fmaf(c, x1.z, o[6]); o[7] = fmaf(c, x1.w, o[7]);
    }
  }
  const int64_t R = (int64_t)a.total_q * a.heads;
  const int64_t row = t * a.heads + h;
  const bool any = tot > 0.f;
  const float inv = any ? 1.f / tot : 0.f;
  const float row_lse = any ? (mx + log2f(tot)) * kLn2 : -INFINITY;
  if (S == 1) {
    uint32_t wv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 v = __floats2bfloat162_rn(o[2 * e] * inv, o[2 * e + 1] * inv);
      wv[e] = *reinterpret_cast<const uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(a.out + row * kDv + d0) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    if (d0 == 0) a.lse[row] = row_lse;
  } else {
    float4* dst = reinterpret_cast<float4*>(a.ws_o + ((int64_t)split * R + row) * kDv + d0);
    dst[0] = make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
    dst[1] = make_float4(o[4] * inv, o[5] * inv, o[6] * inv, o[7] * inv);
    if (d0 == 0) a.ws_lse[(int64_t)split * R + row] = row_lse;
  }
}

static std::once_flag g_simt_attr_once;
static cudaError_t g_simt_attr = cudaSuccess;

cudaError_t launch_verify_simt(const VerifyArgs& a, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  std::call_once(g_simt_attr_once, [] {
    g_simt_attr = cudaFuncSetAttribute(verify_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSimtSmem);
  });
  if (g_simt_attr != cudaSuccess) return g_simt_attr;
  const int hg_count = (a.heads + kRows - 1) / kRows;
  // No request has more keys than kv_indices holds, and a split holds at
  // least kMinKeysY keys, so no request uses more than this many splits:
  // CTAs beyond it would only find that out (after reading the request's
  // geometry) and exit.
  const int64_t need = (a.kv_len + kMinKeysY - 1) / kMinKeysY;
  const int gy = (int)(need < 1 ? 1 : need < a.max_splits ? need : a.max_splits);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)a.total_q * hg_count), (unsigned)gy);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = kSimtSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_simt_kernel, a);
}

// Whether a warp-shuffle call with these host-known sizes may split a
// request (and so needs the merge): only when some request can have more
// keys than one split of the grid takes.
bool simt_may_split(int max_splits, int64_t kv_len) { return max_splits > 1 && kv_len > kMinKeysY; }

// ---------------------------------------------------------------- merge

// lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * o_s  -> bf16.
// One CTA per (token, group of heads). Each thread owns the 16 bytes of an
// fp32 partial row that one vector load brings in (4 dims). The producing
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
  static_assert(kVec == 4, "fp32 partials: 4 dims per 16-byte load");
  *reinterpret_cast<uint2*>(a.out + row * kDv + kVec * dv) = make_uint2(o[0], o[1]);
  if (dv == 0) a.lse[row] = tot > 0.f ? mx + logf(tot) : -INFINITY;
}

cudaError_t launch_lse_merge(const VerifyArgs& a, cudaStream_t stream) {
  // Programmatic dependent launch: the merge grid is scheduled while the
  // producing kernel drains and waits on-device for its completion, which
  // hides the launch gap between the two.
  cudaLaunchConfig_t cfg = {};
  const int heads_per_cta = MergeShape<float>::kHeads;
  cfg.gridDim = dim3((unsigned)a.total_q, (unsigned)((a.heads + heads_per_cta - 1) / heads_per_cta));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lse_merge_kernel<float>, a);
}

}  // namespace mt
