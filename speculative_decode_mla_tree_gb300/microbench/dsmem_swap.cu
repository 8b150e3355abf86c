// Cost of swapping 32 KB between the two CTAs of a cluster: the two CTAs of each cluster
// swap 32 KB per iteration, (A) by 16-byte st.async from 128 threads,
// (B) by local stores + one bulk shared::cta -> shared::cluster copy.
#include <cstdio>
#include "../csrc/sm100_ptx.cuh"
using namespace mt::sm100;
constexpr int kBytes = 32768, kIters = 200;
__device__ int g_abort;

__device__ __forceinline__ void bulk_s2s(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes, uint32_t bar_cluster) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst_cluster), "r"(src_cta), "r"(bytes), "r"(bar_cluster) : "memory");
}

template <int MODE>
__global__ void __launch_bounds__(128, 1) k_x(float* sink) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full, freeb;
  volatile int* ab = &g_abort;
  const int r = threadIdx.x;
  const uint32_t peer = cluster_ctarank() ^ 1;
  float* in = (float*)sm;
  float* out = (float*)(sm + kBytes);
  if (r == 0) { mbar_init(&full, 1); mbar_init(&freeb, 1); fence_mbar_init_cluster(); }
  __syncthreads();
  cluster_sync();
  const uint32_t in_peer = mapa(smem_u32(in), peer);
  const uint32_t full_peer = mapa(smem_u32(&full), peer);
  const uint32_t free_peer = mapa(smem_u32(&freeb), peer);
  float acc = 0.f;
  for (int it = 0; it < kIters; ++it) {
    if (r == 0) mbar_arrive_expect_tx(&full, kBytes);
    mbar_wait<true>(&freeb, (it & 1) ^ 1, ab);           // peer's `in` is free
    if (MODE == 0) {
      for (int c = 0; c < 16; ++c)
        st_async_v4(in_peer + r * 256 + c * 16, r + c, it, 1, 2, full_peer);
    } else {
      for (int c = 0; c < 16; ++c)
        *(uint4*)(out + r * 64 + c * 4) = make_uint4(r + c, it, 1, 2);
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (r == 0) {
        bulk_s2s(in_peer, smem_u32(out), kBytes, full_peer);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    }
    mbar_wait<true>(&full, it & 1, ab);                    // peer's data arrived
    acc += in[r * 64 + (it & 63)];
    if (MODE == 1 && r == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    named_bar_sync(1, 128);
    if (r == 0) mbar_arrive_remote(free_peer);
  }
  cluster_sync();
  if (acc == 12345.f) sink[0] = acc;
}

int main() {
  float* sink; cudaMalloc(&sink, 4);
  cudaFuncSetAttribute(k_x<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * kBytes + 1024);
  cudaFuncSetAttribute(k_x<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * kBytes + 1024);
  cudaLaunchConfig_t cfg = {}; cfg.gridDim = dim3(152); cfg.blockDim = dim3(128); cfg.dynamicSmemBytes = 2 * kBytes + 1024;
  cudaLaunchAttribute at; at.id = cudaLaunchAttributeClusterDimension; at.val.clusterDim.x = 2; at.val.clusterDim.y = 1; at.val.clusterDim.z = 1;
  cfg.attrs = &at; cfg.numAttrs = 1;
  cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
  for (int mode = 0; mode < 2; ++mode) {
    float best = 1e9;
    for (int i = 0; i < 5; ++i) {
      cudaEventRecord(e0);
      if (mode == 0) cudaLaunchKernelEx(&cfg, k_x<0>, sink); else cudaLaunchKernelEx(&cfg, k_x<1>, sink);
      cudaEventRecord(e1); cudaEventSynchronize(e1);
      float ms; cudaEventElapsedTime(&ms, e0, e1); if (ms < best) best = ms;
    }
    printf("%s: %.3f us per 32 KB swap (%s)\n", mode == 0 ? "st.async 16B x 2048" : "local st + bulk copy",
           best * 1e3 / kIters, cudaGetErrorString(cudaGetLastError()));
  }
  int ab = 0; cudaMemcpyFromSymbol(&ab, g_abort, 4); printf("abort flag %d\n", ab);
  return 0;
}
