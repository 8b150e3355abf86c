// Random-row gather rate on this GPU: 152 CTAs, each streams NB blocks of
// 64 random pool rows (576 B per row: 4 x 128 B + 64 B, as one CTA of the
// verify cluster loads) into 2 shared-memory stages.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "../csrc/sm100_ptx.cuh"
using namespace mt::sm100;

constexpr int BN = 64, NB = 64, kStage = 36864;
__device__ int g_abort;

__global__ void __launch_bounds__(128) k_gather4(const __grid_constant__ CUtensorMap lat, const __grid_constant__ CUtensorMap rope,
                                                 const int* slots, int pieces_per_row) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[2];
  volatile int* ab = &g_abort;
  if (threadIdx.x == 0) { mbar_init(&full[0], 1); mbar_init(&full[1], 1); }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int* sl = slots + (size_t)blockIdx.x * NB * BN;
  for (int b = 0; b < NB; ++b) {
    const int s = b & 1;
    if (b >= 2 && lane == 0) mbar_wait<false>(&full[s], ((b - 2) >> 1) & 1, ab);
    if (lane == 0) mbar_arrive_expect_tx(&full[s], pieces_per_row == 5 ? kStage : 4 * 8192);
    __syncwarp();
    if (lane < 16) {
      const int* r = sl + b * BN + 4 * lane;
      int y0 = r[0], y1 = r[1], y2 = r[2], y3 = r[3];
      uint8_t* st = sm + s * kStage;
      for (int k = 0; k < 4; ++k) tma_gather4(st + k * 8192 + lane * 512, &lat, 64 * k, y0, y1, y2, y3, &full[s]);
      if (pieces_per_row == 5) tma_gather4(st + 32768 + lane * 256, &rope, 512, y0, y1, y2, y3, &full[s]);
    }
    __syncwarp();
  }
  if (lane == 0) { mbar_wait<false>(&full[0], ((NB - 2) >> 1) & 1, ab); mbar_wait<false>(&full[1], ((NB - 1) >> 1) & 1, ab); }
}

__global__ void __launch_bounds__(128) k_cpasync(const uint16_t* pool, const int* slots) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
  const int* sl = slots + (size_t)blockIdx.x * NB * BN;
  for (int b = 0; b < NB; ++b) {
    uint8_t* st = sm + (b & 1) * kStage;
    // 64 rows x 36 sixteen-byte pieces = 2304 pieces, 18 per thread
    for (int i = threadIdx.x; i < BN * 36; i += 128) {
      const int row = i / 36, piece = i % 36;
      const char* src = (const char*)(pool + (size_t)sl[b * BN + row] * 576) + (piece < 32 ? piece * 16 : 1024 + (piece - 32) * 16);
      uint32_t dst = smem_u32(st + row * 576 + piece * 16);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

__global__ void __launch_bounds__(128) k_tile(const __grid_constant__ CUtensorMap lat) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[2];
  volatile int* ab = &g_abort;
  if (threadIdx.x == 0) { mbar_init(&full[0], 1); mbar_init(&full[1], 1); }
  __syncthreads();
  if (threadIdx.x != 0) return;
  for (int b = 0; b < NB; ++b) {
    const int s = b & 1;
    if (b >= 2) mbar_wait<false>(&full[s], ((b - 2) >> 1) & 1, ab);
    mbar_arrive_expect_tx(&full[s], 4 * 8192);
    const int y = (blockIdx.x * NB + b) * BN;  // contiguous rows
    for (int k = 0; k < 4; ++k) tma_load_2d(sm + s * kStage + k * 8192, &lat, 64 * k, y, &full[s]);
  }
  mbar_wait<false>(&full[0], ((NB - 2) >> 1) & 1, ab);
  mbar_wait<false>(&full[1], ((NB - 1) >> 1) & 1, ab);
}

static PFN_cuTensorMapEncodeTiled_v12000 enc() {
  void* fn = nullptr; cudaDriverEntryPointQueryResult q;
  cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  return (PFN_cuTensorMapEncodeTiled_v12000)fn;
}
static CUtensorMap map(void* base, uint64_t rows, uint32_t bc, uint32_t br, CUtensorMapSwizzle sw) {
  CUtensorMap m; cuuint64_t d[2] = {576, rows}; cuuint64_t st[1] = {1152}; cuuint32_t bx[2] = {bc, br}; cuuint32_t es[2] = {1, 1};
  CUresult r = enc()(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) { printf("encode failed %d\n", (int)r); exit(1); }
  return m;
}

int main() {
  const uint64_t rows = 1 << 20;  // 1.2 GB pool: far larger than L2
  const int ctas = 152;
  uint16_t* pool; int* slots;
  cudaMalloc(&pool, rows * 1152); cudaMemset(pool, 0, rows * 1152);
  std::vector<int> h((size_t)ctas * NB * BN);
  srand(1); for (auto& x : h) x = (int)(((uint64_t)rand() * 7919u) % rows);
  cudaMalloc(&slots, h.size() * 4); cudaMemcpy(slots, h.data(), h.size() * 4, cudaMemcpyHostToDevice);
  CUtensorMap lat = map(pool, rows, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B);
  CUtensorMap rope = map(pool, rows, 32, 1, CU_TENSOR_MAP_SWIZZLE_64B);
  CUtensorMap tile = map(pool, rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  const int smem = 2 * kStage + 1024;
  cudaFuncSetAttribute(k_gather4, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaFuncSetAttribute(k_cpasync, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaFuncSetAttribute(k_tile, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
  auto run = [&](const char* name, double bytes, auto launch) {
    launch(); cudaDeviceSynchronize();
    float best = 1e9;
    for (int i = 0; i < 5; ++i) { cudaEventRecord(e0); launch(); cudaEventRecord(e1); cudaEventSynchronize(e1); float ms; cudaEventElapsedTime(&ms, e0, e1); if (ms < best) best = ms; }
    printf("%-34s %8.1f us  %8.1f GB/s  (%s)\n", name, best * 1e3, bytes / (best * 1e-3) / 1e9, cudaGetErrorString(cudaGetLastError()));
  };
  const double b576 = (double)ctas * NB * BN * 576, b512 = (double)ctas * NB * BN * 512;
  run("gather4 5 pieces/row (576 B)", b576, [&] { k_gather4<<<ctas, 128, smem>>>(lat, rope, slots, 5); });
  run("gather4 4 pieces/row (512 B)", b512, [&] { k_gather4<<<ctas, 128, smem>>>(lat, rope, slots, 4); });
  run("cp.async 16 B, 128 thr (576 B)", b576, [&] { k_cpasync<<<ctas, 128, smem>>>(pool, slots); });
  run("tile loads contiguous (512 B)", b512, [&] { k_tile<<<ctas, 128, smem>>>(tile); });
  int ab = 0; cudaMemcpyFromSymbol(&ab, g_abort, 4); printf("abort flag %d\n", ab);
  return 0;
}
