// TMA tile::gather4 issue rate versus the number of issuing warps in one CTA.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <functional>
#include <vector>
#include "../csrc/sm100_ptx.cuh"
using namespace mt::sm100;

constexpr int BN = 64, NB = 48, ROWB = 1152;
constexpr int kStageB = BN * ROWB;
__device__ int g_abort;

// W producer warps; warp w gathers rows [w*BN/W, (w+1)*BN/W) of every block (4 rows per lane)
__global__ void k_g4w(const __grid_constant__ CUtensorMap m, const int* slots, int W, int stages, int lat_pieces) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[8];
  volatile int* ab = &g_abort;
  if (threadIdx.x < 8) mbar_init(&full[threadIdx.x], W);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= W) return;
  const int lanes = 16 / W;               // gather lanes per warp
  const int piece_b = 128;
  const int stage_bytes = BN * lat_pieces * piece_b;
  const int* sl = slots + (size_t)blockIdx.x * NB * BN;
  for (int b = 0; b < NB; ++b) {
    const int s = b % stages;
    if (b >= stages && lane == 0) mbar_wait<false>(&full[s], ((b - stages) / stages) & 1, ab);
    if (lane == 0) mbar_arrive_expect_tx(&full[s], stage_bytes / W);
    __syncwarp();
    if (lane < lanes) {
      const int g = warp * lanes + lane;  // 4-row group of the block
      const int* r = sl + b * BN + 4 * g;
      int y0 = r[0], y1 = r[1], y2 = r[2], y3 = r[3];
      uint8_t* st = sm + s * stage_bytes;
      for (int k = 0; k < lat_pieces; ++k)
        tma_gather4(st + k * BN * piece_b + g * 4 * piece_b, &m, 64 * k, y0, y1, y2, y3, &full[s]);
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
  uint8_t* pool; int* slots; uint8_t* flush;
  cudaMalloc(&pool, rows * ROWB); cudaMemset(pool, 1, rows * ROWB);
  cudaMalloc(&flush, 512ull << 20);
  const size_t n = (size_t)152 * NB * BN;
  std::vector<int> h(n);
  srand(3); for (auto& x : h) x = (int)((((uint64_t)rand() << 31) ^ (uint64_t)rand()) % rows);
  cudaMalloc(&slots, n * 4); cudaMemcpy(slots, h.data(), n * 4, cudaMemcpyHostToDevice);
  CUtensorMap m; cuuint64_t d[2] = {576, rows}; cuuint64_t st[1] = {ROWB}; cuuint32_t bx[2] = {64, 1}; cuuint32_t es[2] = {1, 1};
  enc()(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pool, d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  cudaFuncSetAttribute(k_g4w, cudaFuncAttributeMaxDynamicSharedMemorySize, 226 * 1024);
  cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
  auto run = [&](const char* nm, double bytes, std::function<void()> launch) {
    float best = 1e9;
    for (int i = 0; i < 6; ++i) {
      cudaMemsetAsync(flush, i, 512ull << 20);
      cudaEventRecord(e0); launch(); cudaEventRecord(e1);
      cudaEventSynchronize(e1); float ms; cudaEventElapsedTime(&ms, e0, e1);
      if (i > 0) best = std::min(best, ms);
    }
    printf("%-44s %8.1f us  %8.1f GB/s  (%s)\n", nm, best * 1e3, bytes / (best * 1e-3) / 1e9, cudaGetErrorString(cudaGetLastError()));
  };
  for (int pieces : {9, 4}) {
    const double bytes = 152.0 * NB * BN * pieces * 128;
    const int sm2 = 2 * BN * pieces * 128 + 1024, sm3 = 3 * BN * pieces * 128 + 1024;
    char nm[96];
    for (int W : {1, 2, 4, 8}) {
      snprintf(nm, sizeof nm, "%d x128B pieces, %d warps, 2 stages", pieces, W);
      run(nm, bytes, [&] { k_g4w<<<152, 32 * W, sm2>>>(m, slots, W, 2, pieces); });
    }
    snprintf(nm, sizeof nm, "%d x128B pieces, 4 warps, 3 stages", pieces);
    if (sm3 <= 226 * 1024) run(nm, bytes, [&] { k_g4w<<<152, 128, sm3>>>(m, slots, 4, 3, pieces); });
  }
  int ab = 0; cudaMemcpyFromSymbol(&ab, g_abort, 4); printf("abort flag %d\n", ab);
  return 0;
}
