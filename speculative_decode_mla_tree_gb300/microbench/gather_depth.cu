// Random-row gather rate versus stages in flight, piece size and slot order.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "../csrc/sm100_ptx.cuh"
using namespace mt::sm100;

constexpr int BN = 64, NB = 48;
__device__ int g_abort;

// Each CTA streams NB blocks of 64 rows; per row `pieces` gathers of 128 B
// (columns 64k, k < pieces), through `stages` buffers of 64 x pieces x 128 B.
__global__ void __launch_bounds__(128) k_g(const __grid_constant__ CUtensorMap lat, const int* slots,
                                           int pieces, int stages, int col_off) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[8];
  volatile int* ab = &g_abort;
  if (threadIdx.x < 8) mbar_init(&full[threadIdx.x], 1);
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int stage_bytes = BN * pieces * 128;
  const int* sl = slots + (size_t)blockIdx.x * NB * BN;
  for (int b = 0; b < NB; ++b) {
    const int s = b % stages;
    if (b >= stages && lane == 0) mbar_wait<false>(&full[s], ((b - stages) / stages) & 1, ab);
    if (lane == 0) mbar_arrive_expect_tx(&full[s], stage_bytes);
    __syncwarp();
    if (lane < 16) {
      const int* r = sl + b * BN + 4 * lane;
      int y0 = r[0], y1 = r[1], y2 = r[2], y3 = r[3];
      uint8_t* st = sm + s * stage_bytes;
      for (int k = 0; k < pieces; ++k)
        tma_gather4(st + k * BN * 128 + lane * 512, &lat, col_off + 64 * k, y0, y1, y2, y3, &full[s]);
    }
    __syncwarp();
  }
  if (lane == 0)
    for (int b = NB - stages; b < NB; ++b) mbar_wait<false>(&full[b % stages], (b / stages) & 1, ab);
}

static PFN_cuTensorMapEncodeTiled_v12000 enc() {
  void* fn = nullptr; cudaDriverEntryPointQueryResult q;
  cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  return (PFN_cuTensorMapEncodeTiled_v12000)fn;
}

int main() {
  const uint64_t rows = 1 << 20;
  const int ctas = 152;
  uint16_t* pool; int* slots; int* sorted;
  cudaMalloc(&pool, rows * 1152); cudaMemset(pool, 0, rows * 1152);
  std::vector<int> h((size_t)ctas * NB * BN);
  srand(1); for (auto& x : h) x = (int)(((uint64_t)rand() * 7919u) % rows);
  cudaMalloc(&slots, h.size() * 4); cudaMemcpy(slots, h.data(), h.size() * 4, cudaMemcpyHostToDevice);
  for (size_t i = 0; i < h.size(); i += BN) std::sort(h.begin() + i, h.begin() + i + BN);
  cudaMalloc(&sorted, h.size() * 4); cudaMemcpy(sorted, h.data(), h.size() * 4, cudaMemcpyHostToDevice);
  CUtensorMap m; cuuint64_t d[2] = {576, rows}; cuuint64_t st[1] = {1152}; cuuint32_t bx[2] = {64, 1}; cuuint32_t es[2] = {1, 1};
  enc()(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pool, d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  cudaFuncSetAttribute(k_g, cudaFuncAttributeMaxDynamicSharedMemorySize, 226 * 1024);
  cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
  struct Cfg { int pieces, stages, col; const int* sl; const char* nm; };
  Cfg cfgs[] = {{4, 2, 0, slots, "half row 512B, 2 stages"}, {4, 4, 0, slots, "half row 512B, 4 stages"},
                {4, 6, 0, slots, "half row 512B, 6 stages"}, {9, 1, 0, slots, "full row 1152B, 1 stage"},
                {9, 2, 0, slots, "full row 1152B, 2 stages"}, {9, 3, 0, slots, "full row 1152B, 3 stages"},
                {4, 4, 0, sorted, "half row 512B, 4 st, sorted"}, {9, 2, 0, sorted, "full row, 2 st, sorted"}};
  for (auto& c : cfgs) {
    const int smem = c.stages * BN * c.pieces * 128 + 1024;
    if (smem > 226 * 1024) { printf("%s: too big\n", c.nm); continue; }
    k_g<<<ctas, 128, smem>>>(m, c.sl, c.pieces, c.stages, c.col); cudaDeviceSynchronize();
    float best = 1e9;
    for (int i = 0; i < 5; ++i) {
      cudaEventRecord(e0); k_g<<<ctas, 128, smem>>>(m, c.sl, c.pieces, c.stages, c.col); cudaEventRecord(e1);
      cudaEventSynchronize(e1); float ms; cudaEventElapsedTime(&ms, e0, e1); best = std::min(best, ms);
    }
    const double bytes = (double)ctas * NB * BN * c.pieces * 128;
    printf("%-32s %8.1f us  %8.1f GB/s  (%s)\n", c.nm, best * 1e3, bytes / (best * 1e-3) / 1e9, cudaGetErrorString(cudaGetLastError()));
  }
  int ab = 0; cudaMemcpyFromSymbol(&ab, g_abort, 4); printf("abort flag %d\n", ab);
  return 0;
}
