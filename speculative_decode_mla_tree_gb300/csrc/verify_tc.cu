// Tensor-core (tcgen05 / TMEM) tree-verify attention for sm_103a.
//
// What it computes is the verify call of "The Moment of Truth: Flipping the
// Switch on a Custom CUDA Verify Kernel" (section "The Long Road to Parity":
// prefix + draft KV gathered through kv_indices, mask row stride prefix +
// draft) with the split-KV flash-decode structure of its section "The
// Broader Context", on the absorbed MLA shapes of "The Pivot to Live
// Cutover" (section "Input Knowledge Required": 512 latent + 64 rope dims).
// The pages' sm_120 kernel (no TMA, no tcgen05, 100 KB of shared memory) is
// prior art; this kernel is laid out for GB300 instead.
//
// Work item: one 128-row tile of a request's (draft node, head) rows and one
// contiguous range of its key positions (a split). A tile is served by a
// cluster of two CTAs on two SMs that split the head dims: CTA c holds
// latent dims [256c, 256c+256) and rope dims [512+32c, 512+32c+32) of the
// query tile and of every key row. Per block of BN = 48 key rows:
//
//   query     per item: the rope half by TMA into shared memory, the
//             256 latent dims by the sender warps straight into TMEM
//   TMA       key-row halves by tile::gather4 through kv_indices, four rows
//             per instruction, five stages in flight
//   tcgen05   S_c = Q_c K_c^T   (M=128, N=48, K=288) into TMEM
//   DSMEM     each CTA rounds its partial S_c (scaled to the log2
//             domain) to fp16 and sends it to its peer; both form
//             fp16(S_0) + fp16(S_1) in fp32, so both hold bit-identical S
//   softmax   mask bytes staged per block as bits, online max / sum in the
//             log2 domain with lazy rescaling (the running max moves only
//             when it grows by more than 8, i.e. a factor of 256)
//   tcgen05   O_c += P V_c      (M=128, N=256, K=48) into TMEM; V_c is the
//             same shared-memory key tile, read MN-major
//
// Why two CTAs: a 128-row fp32 accumulator for all 512 value dims is the
// whole 256 KB of TMEM. Splitting the dims halves it and leaves TMEM room
// for the query's latent half (so the QK MMAs read no query bytes from
// shared memory, which at N = 48 would otherwise bound them) and two score
// buffers; the exchange stays at the 48-column score block.
//
// Roles per CTA (384 threads): warps 0-3 softmax / epilogue (one thread per
// TMEM lane = tile row), warps 4-7 score senders (same lanes), warps 8-10
// TMA producers (one warp alone issues tile::gather4 too slowly to keep
// up), warp 11 MMA issuer
// and TMEM owner. Every mbarrier wait is time-bounded: a timeout sets
// MT_DEV_TIMEOUT, after which the CTA runs through to its exit without
// waiting, draining its asynchronous copies and MMAs before releasing TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include <cuda_fp16.h>

#include "mt_common.cuh"
#include "mt_internal.h"
#include "sm100_ptx.cuh"

namespace mt {
namespace tc {

using namespace sm100;

constexpr int BM = 128;          // tile rows = TMEM lanes
constexpr int BN = 48;           // key rows per block
constexpr int kGatherLanes = BN / 4;  // four-row groups per block (tile::gather4)
constexpr int kProducers = 3;    // TMA producer warps (one warp issues about 37 ns per gather4)
constexpr int kFirstProducer = 8;  // warps 0-3 softmax, 4-7 score senders
constexpr int kMmaWarp = kFirstProducer + kProducers;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr int kMaxBatch = 256;
constexpr float kRescale = 8.f;  // lazy-rescale threshold (log2 units)
constexpr int kMinChunk = 256;   // smallest split worth a work item (key rows)
constexpr int kMaskPrefetch = 2; // mask (node, group) pairs per thread held one block ahead
constexpr int kSlotAhead = 2;    // key blocks whose slot numbers are in flight ahead of the gathers
constexpr int kWarmBlocks = 512; // most key blocks per cluster (upper bound) for the dry-pass variant

// Shared memory map (offsets from a 1024-byte aligned base).
constexpr int kQRope = 0;                             // query rope half [128 rows x 64 B], 64B swizzle
constexpr int kKV = kQRope + BM * 64;                 // key stages
constexpr int kKVLat = BN * 128;                      // one latent chunk of a stage
constexpr int kKVStage = 4 * kKVLat + BN * 64;        // 27648
constexpr int kStages = 5;
constexpr int kX = kKV + kStages * kKVStage;          // exchange: [XO0 | XP0 | XO1 | XP1]
constexpr int kXRow = BN * 2 + 16;                    // fp16 scores of one row, padded: rows land on different banks
constexpr int kXBytes = BM * kXRow;                   // one buffer (own XO or peer's XP)
constexpr int kVisNodes = BM + 2;                     // distinct draft nodes a tile can touch
constexpr int kVis = kX + 4 * kXBytes;                // 2 x kVisNodes x 64-bit masks
constexpr int kBars = kVis + 2 * kVisNodes * 8;
constexpr int B_Q_FULL = 0;                     // query rope half landed (TMA)
constexpr int B_QT_FULL = 1;                    // query latent half written to TMEM
constexpr int B_Q_EMPTY = 2;                    // last QK of the item done
constexpr int B_KV_FULL0 = 3;                   // kStages barriers each
constexpr int B_KV_EMPTY0 = B_KV_FULL0 + kStages;
constexpr int B_S_FULL0 = B_KV_EMPTY0 + kStages;  // two each from here
constexpr int B_S_EMPTY0 = B_S_FULL0 + 2;
constexpr int B_X_FULL0 = B_S_EMPTY0 + 2;
constexpr int B_X_FREE0 = B_X_FULL0 + 2;
constexpr int B_P_FULL = B_X_FREE0 + 2;
constexpr int B_O_DONE = B_P_FULL + 1;
constexpr int B_O_FREE = B_O_DONE + 1;
constexpr int B_DRAIN = B_O_FREE + 1;
constexpr int kNumBars = B_DRAIN + 1;
constexpr int kMisc = kBars + kNumBars * 8;           // tmem base, abort flag, item count, B_DRY
constexpr int B_DRY = (kMisc + 16 - kBars) / 8;       // never completes: the dry passes' waits and signals
constexpr int kPlan = kMisc + 32;                     // per-request plan
constexpr int kPlanStride = 9;                        // int32 words per request
constexpr int kOrd = kPlan + kMaxBatch * kPlanStride * 4;   // request at each rank
constexpr int kOBase = kOrd + kMaxBatch * 4;          // first item of each rank (+ total)
constexpr int kSmemUsed = kOBase + (kMaxBatch + 1) * 4;
constexpr int kSmemBytes = kSmemUsed + 1024;          // slack for aligning the base
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kMisc % 8 == 0 && kBars + 8 * B_DRY + 8 <= kPlan, "B_DRY sits in the misc area");
static_assert(2 * kXBytes >= BM * 128, "epilogue staging fits in one XO/XP pair");
static_assert(BN % 16 == 0 && BN <= 64, "block width");
static_assert(kQRope % 1024 == 0 && kKV % 1024 == 0 && kX % 1024 == 0 &&
                  kKVStage % 1024 == 0 && kBars % 8 == 0,
              "alignment");

constexpr uint32_t kQTx = BM * 64;                    // query rope bytes per CTA per item
constexpr uint32_t kKVTx = kKVStage;                  // key bytes per CTA per block
constexpr uint32_t kTmemCols = 512;
// TMEM columns (512 x 128 lanes; lane = tile row):
//   [0, 256)    O, this CTA's 256 value dims (fp32)
//   [256, 384)  Q, this CTA's 256 latent query dims as bf16 pairs: QK's A
//               operand (no shared-memory reads of Q per MMA)
//   [384, 432)  S buffer 0, [448, 496) S buffer 1 (BN fp32 scores each)
//   P (bf16 pairs, PV's A), one 8-column piece per 16 keys, in the gaps:
//   [432, 448) and [496, 504)
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemQ = 256;
constexpr uint32_t kTmemS = 384;                      // buffer b at kTmemS + 64 b
__host__ __device__ constexpr uint32_t tmem_p_col(int t) { return t < 2 ? 432u + 8u * t : 496u; }
static_assert(BN == 48, "TMEM map holds 48-column score blocks and three P pieces");
constexpr uint64_t kDrainNs = 100000000ull;           // 100 ms
constexpr long long kIdleLimitCycles = 4000000000ll;  // about 2 s of SM clock with nothing to issue

// plan words
enum { PL_Q0, PL_N, PL_KV0, PL_L, PL_SPLITS, PL_LEN, PL_TILES, PL_M0LO, PL_M0HI };

struct TcParams {
  VerifyArgs a;
  int nclusters;
};

struct Item {
  int b, tile, split, splits;
  int q0, n, kv0, L, j0, j1, nblocks, row0;
  int64_t mask0;
};

// Item numbering: requests are ranked (longest split first when the items
// take more than one round of the persistent grid), a request's items are
// numbered tile-major, and cluster c takes item k * nclusters + c in even
// rounds k and k * nclusters + (nclusters - 1 - c) in odd ones, so the
// longest items are spread over the clusters first and every cluster's
// total comes out close to the mean.
__device__ __forceinline__ int item_of(int k, int c, int nclusters) {
  return k * nclusters + ((k & 1) ? nclusters - 1 - c : c);
}

__device__ __forceinline__ Item decode_item(const int* plan, const int* ord, const int* obase,
                                            int batch, int id) {
  int lo = 0, hi = batch - 1;  // last rank whose first item is <= id
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (obase[mid] <= id) lo = mid; else hi = mid - 1;
  }
  const int b = ord[lo];
  const int* pr = plan + b * kPlanStride;
  Item it;
  it.b = b;
  it.q0 = pr[PL_Q0];
  it.n = pr[PL_N];
  it.kv0 = pr[PL_KV0];
  it.L = pr[PL_L];
  it.splits = pr[PL_SPLITS];
  const int len = pr[PL_LEN];
  const int local = id - obase[lo];
  it.tile = local / it.splits;
  it.split = local - it.tile * it.splits;
  it.j0 = it.split * len;
  it.j1 = min(it.L, it.j0 + len);
  it.nblocks = (it.j1 - it.j0 + BN - 1) / BN;
  it.row0 = it.tile * BM;
  it.mask0 = (int64_t)(uint32_t)pr[PL_M0LO] | ((int64_t)pr[PL_M0HI] << 32);
  return it;
}

__device__ __forceinline__ long long warp_sum(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Warp 0: per-request geometry, split counts and the item numbering. Every
// CTA computes the same plan from the device indptrs; one CTA also publishes
// the split counts for the merge kernel.
//
// Split length: a quarter of one cluster's fair share of (tile x key) work,
// at least kMinChunk keys, so that a long request is cut into enough items
// for every cluster to get several and the last round stays short.
__device__ void build_plan(const VerifyArgs& a, int nclusters, int* plan, int* ord, int* obase,
                           int* total_items, int lane, bool publish) {
  const int H = a.heads;
  long long units = 0;
  for (int b = lane; b < a.batch; b += 32) {
    const ReqGeom g = request_geom(a.kv_indptr, a.qo_indptr, a.mask_indptr, b, a.kv_len,
                                   a.mask_len, a.total_q, a.bits_mask != 0);
    int* pr = plan + b * kPlanStride;
    int tiles = 0;
    if (g.ok && g.n > 0) tiles = (int)(((long long)g.n * H + BM - 1) / BM);
    if (!g.ok && publish) flag(a.status, MT_DEV_BAD_INDPTR);
    pr[PL_Q0] = (int)g.q0;
    pr[PL_N] = g.n;
    pr[PL_KV0] = (int)g.kv0;
    pr[PL_L] = g.L;
    pr[PL_TILES] = tiles;
    pr[PL_M0LO] = (int)(uint32_t)(g.mask0 & 0xffffffffLL);
    pr[PL_M0HI] = (int)(g.mask0 >> 32);
    units += (long long)tiles * g.L;
  }
  units = warp_sum(units);
  const long long nc = nclusters > 0 ? nclusters : 1;
  long long chunk = (units + 4 * nc - 1) / (4 * nc);
  if (chunk < kMinChunk) chunk = kMinChunk;
  chunk = (chunk + BN - 1) / BN * BN;
  long long items_total = 0;
  for (int b = lane; b < a.batch; b += 32) {
    int* pr = plan + b * kPlanStride;
    const int tiles = pr[PL_TILES];
    const int L = pr[PL_L];
    int S = 1, len = BN;
    if (tiles > 0 && L > 0) {
      long long s = (L + chunk - 1) / chunk;
      if (s > a.max_splits) s = a.max_splits;
      if (s < 1) s = 1;
      len = (int)(((L + s - 1) / s + BN - 1) / BN * BN);
      S = (L + len - 1) / len;
    }
    pr[PL_SPLITS] = S;
    pr[PL_LEN] = len;
    items_total += (long long)tiles * S;
    if (publish) {  // every token of this request: its split count for the merge
      const int q0 = pr[PL_Q0], n = tiles > 0 ? pr[PL_N] : 0;
      for (int tk = 0; tk < n; ++tk) a.ws_tok[q0 + tk] = S;
    }
  }
  items_total = warp_sum(items_total);
  __syncwarp();
  // rank the requests: by split length, longest first, when the items take
  // more than one round; else in request order
  const bool sorted = items_total > nc;
  for (int b = lane; b < a.batch; b += 32) {
    int rank = b;
    if (sorted) {
      const int* pb = plan + b * kPlanStride;
      const int key = pb[PL_TILES] > 0 ? pb[PL_LEN] : -1;
      rank = 0;
      for (int o = 0; o < a.batch; ++o) {
        const int* po = plan + o * kPlanStride;
        const int ko = po[PL_TILES] > 0 ? po[PL_LEN] : -1;
        rank += (ko > key) || (ko == key && o < b);
      }
    }
    ord[rank] = b;
  }
  __syncwarp();
  int carry = 0;
  for (int base = 0; base < a.batch; base += 32) {
    const int r = base + lane;
    int items = 0;
    if (r < a.batch) {
      const int* pr = plan + ord[r] * kPlanStride;
      items = pr[PL_TILES] * pr[PL_SPLITS];
    }
    int incl = items;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (r < a.batch) obase[r] = carry + incl - items;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  // tokens of inconsistent requests (or outside every request) are not merged
  if (publish) {
    __syncwarp();
    for (int tk = lane; tk < a.total_q; tk += 32) {
      int covered = 0;
      for (int b = 0; b < a.batch && !covered; ++b) {
        const int* pr = plan + b * kPlanStride;
        covered = pr[PL_TILES] > 0 && tk >= pr[PL_Q0] && tk < pr[PL_Q0] + pr[PL_N];
      }
      if (!covered) a.ws_tok[tk] = 0;
    }
  }
  if (lane == 0) {
    obase[a.batch] = carry;
    *total_items = carry;
  }
}

// kBits: the tree mask is in the bit form (rows of ceil(L / 32) words)
// kWarm: dry passes that load the softmax and sender loops' code before the
// first scores arrive (worth it when each cluster has few blocks to do)
// kSkip: prefix columns are visible and their mask entries are not read
template <bool kBits, bool kWarm, bool kSkip>
__global__ void __launch_bounds__(kThreads, 1)
    verify_tc_kernel(const __grid_constant__ TcParams p,
                     const __grid_constant__ CUtensorMap tm_qrope,
                     const __grid_constant__ CUtensorMap tm_kvlat,
                     const __grid_constant__ CUtensorMap tm_kvrope) {
  static_assert(kBits || !kWarm, "the softmax dry pass reads the bit-form mask");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const VerifyArgs& a = p.a;
  const int H = a.heads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t cta = cluster_ctarank();
  const uint32_t peer = cta ^ 1u;
  const int cluster_id = blockIdx.x >> 1;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + kMisc + 4);
  int* total_items_s = reinterpret_cast<int*>(sm + kMisc + 8);
  int* plan = reinterpret_cast<int*>(sm + kPlan);
  int* ord = reinterpret_cast<int*>(sm + kOrd);
  int* obase = reinterpret_cast<int*>(sm + kOBase);
  uint64_t* vis = reinterpret_cast<uint64_t*>(sm + kVis);

  if (tid == 0) {
    mbar_init(&bars[B_Q_FULL], 1);
    mbar_init(&bars[B_QT_FULL], 128);
    mbar_init(&bars[B_Q_EMPTY], 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[B_KV_FULL0 + s], 1);
      mbar_init(&bars[B_KV_EMPTY0 + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[B_S_FULL0 + s], 1);
      mbar_init(&bars[B_S_EMPTY0 + s], 128);
    }
    mbar_init(&bars[B_P_FULL], 128);
    mbar_init(&bars[B_O_DONE], 1);
    mbar_init(&bars[B_O_FREE], 128);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars[B_X_FULL0 + x], 128);  // own senders (one with expect_tx) + the peer's bytes
      mbar_init(&bars[B_X_FREE0 + x], 8);    // own four softmax warps and the peer's, one arrival each
    }
    mbar_init(&bars[B_DRAIN], 1);
    if (kWarm) mbar_init(&bars[B_DRY], (1 << 20) - 1);  // the largest count: its first phase never completes
    *abort = 0;
    fence_mbar_init_cluster();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kFirstProducer && lane == 0) {
    prefetch_tmap(&tm_qrope);
    prefetch_tmap(&tm_kvlat);
    prefetch_tmap(&tm_kvrope);
  }
  // the last CTA publishes the split counts: with fewer items than clusters it
  // has none of its own, so the extra stores delay no item
  // Launched as a programmatic dependent of the kernel before it (the
  // marshaling of the same step): the set-up above overlaps that kernel's
  // tail; nothing it writes is read before it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (warp == 0)
    build_plan(a, p.nclusters, plan, ord, obase, total_items_s, lane, blockIdx.x == gridDim.x - 1);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The peer's barriers must exist before anyone touches them remotely: every
  // thread arrives here, and only the softmax warps (the only ones that
  // reach into the peer) wait before their first remote access.
  cluster_arrive();
  const uint32_t tmem = *tmem_slot;
  const int total_items = *total_items_s;

  if (warp >= kFirstProducer && warp < kFirstProducer + kProducers) {
    // ------------------------------------------------------------ producers
    // kProducers warps share every block's gathers: warp pw issues the
    // four-row groups [pw * kGroupsPerWarp, (pw + 1) * kGroupsPerWarp), one
    // group per lane. The first producer warp also loads the query tile and
    // arms each stage's barrier with the whole stage's byte count (bytes of
    // the other warps may land before that arrival; the phase cannot
    // complete without it).
    constexpr int kGroupsPerWarp = kGatherLanes / kProducers;
    static_assert(kGatherLanes % kProducers == 0, "groups per producer warp");
    const int pw = warp - kFirstProducer;
    const int grp = pw * kGroupsPerWarp + lane;
    const bool gathers = lane < kGroupsPerWarp;
    uint32_t kb = 0, qi = 0;
    const int oob = (int)a.num_slots;  // an out-of-range row: TMA fills zeros
    // Slots of the four key rows of this lane's group in block blk of an
    // item: the loads are only issued here (bit e of `live` marks a position
    // inside the split); the values are checked by take_rows when their
    // gathers are issued, so the load latency stays hidden.
    auto load_rows = [&](const Item& it, int blk, int (&rows)[4], int& live) {
      const int pos0 = it.j0 + blk * BN + 4 * grp;
      live = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        rows[e] = oob;
        if (pos0 + e < it.j1) {
          rows[e] = __ldg(a.kv_indices + it.kv0 + pos0 + e);
          live |= 1 << e;
        }
      }
    };
    // Range-check loaded slots: a bad one is flagged and gathered as an
    // out-of-range row (zeros).
    auto take_rows = [&](const int (&raw)[4], int live, int (&rows)[4]) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int slot = oob;
        if ((live >> e) & 1) {
          const int v = raw[e];
          if (v >= 0 && v < a.num_slots) slot = v;
          else flag(a.status, MT_DEV_BAD_SLOT);
        }
        rows[e] = slot;
      }
    };
    for (int rnd = 0, id = item_of(0, cluster_id, p.nclusters); id < total_items;
         id = item_of(++rnd, cluster_id, p.nclusters)) {
      const Item it = decode_item(plan, ord, obase, a.batch, id);
      const int qrow = it.q0 * H + it.row0;
      if (pw == 0 && lane == 0) {
        mbar_wait<false>(&bars[B_Q_EMPTY], (qi & 1) ^ 1, abort);
        mbar_arrive_expect_tx(&bars[B_Q_FULL], kQTx);
        tma_load_2d(sm + kQRope, &tm_qrope, 512 + 32 * (int)cta, qrow, &bars[B_Q_FULL]);
      }
      ++qi;
      // Slot numbers run kSlotAhead blocks ahead of the gathers. The block
      // loop is unrolled by kSlotAhead so that ring entry u always holds the
      // slots of blocks u, u + kSlotAhead, ...: an entry is reloaded right
      // after its gathers are issued and is not touched again until its
      // block comes up (moving an entry whose load is still in flight would
      // wait for it).
      int ring[kSlotAhead][4], live[kSlotAhead];
#pragma unroll
      for (int d = 0; d < kSlotAhead; ++d) {
#pragma unroll
        for (int e = 0; e < 4; ++e) ring[d][e] = oob;
        live[d] = 0;
        if (gathers && d < it.nblocks) load_rows(it, d, ring[d], live[d]);
      }
      for (int blk0 = 0; blk0 < it.nblocks; blk0 += kSlotAhead) {
#pragma unroll
        for (int u = 0; u < kSlotAhead; ++u) {
          const int blk = blk0 + u;
          if (blk < it.nblocks) {
            const int s = kb % kStages;
            uint8_t* st = sm + kKV + s * kKVStage;
            if (lane == 0) {
              mbar_wait<false>(&bars[B_KV_EMPTY0 + s], ((kb / kStages) & 1) ^ 1, abort);
              if (pw == 0) mbar_arrive_expect_tx(&bars[B_KV_FULL0 + s], kKVTx);
            }
            __syncwarp();
            if (gathers) {
              int rows[4];
              take_rows(ring[u], live[u], rows);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                tma_gather4(st + k * kKVLat + grp * 512, &tm_kvlat, 256 * (int)cta + 64 * k,
                            rows[0], rows[1], rows[2], rows[3], &bars[B_KV_FULL0 + s]);
              tma_gather4(st + 4 * kKVLat + grp * 256, &tm_kvrope, 512 + 32 * (int)cta, rows[0],
                          rows[1], rows[2], rows[3], &bars[B_KV_FULL0 + s]);
              live[u] = 0;
              if (blk + kSlotAhead < it.nblocks) load_rows(it, blk + kSlotAhead, ring[u], live[u]);
            }
            __syncwarp();
            ++kb;
          }
        }
      }
    }
    if (pw == 0 && lane == 0) {  // every copy this CTA issued has landed before it may exit
      if (qi > 0) mbar_drain(&bars[B_Q_FULL], (qi - 1) & 1, kDrainNs);
      for (uint32_t k = kb >= kStages ? kb - kStages : 0; k < kb; ++k)
        mbar_drain(&bars[B_KV_FULL0 + (k % kStages)], (k / kStages) & 1, kDrainNs);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t kb = 0, sc = 0, pc = 0, qi = 0, ii = 0;
      const uint32_t idesc_qk = idesc_bf16(BM, BN, 0, 0);
      const uint32_t idesc_pv = idesc_bf16(BM, 256, 0, 1);
      const uint32_t qrope = smem_u32(sm + kQRope);
      const uint32_t kvbase = smem_u32(sm + kKV);
      for (int rnd = 0, id = item_of(0, cluster_id, p.nclusters); id < total_items;
         id = item_of(++rnd, cluster_id, p.nclusters)) {
        const Item it = decode_item(plan, ord, obase, a.batch, id);
        mbar_wait<false>(&bars[B_Q_FULL], qi & 1, abort);
        mbar_wait<false>(&bars[B_QT_FULL], qi & 1, abort);
        ++qi;
        tc_fence_after();
        const uint32_t kb0 = kb;
        // Two independent streams, polled without blocking: S_j = Q K_j^T
        // as soon as key block j has landed and a score buffer is free
        // (both are read by the senders early), and O += P_j V_j as soon as
        // the softmax has written P_j. Waiting for P_j before issuing the
        // next scores would tie every block to the softmax two blocks back.
        int nq = 0, np = 0;
        bool ofree = false;
        long long idle_since = 0;
        while (np < it.nblocks) {
          bool did = false;
          if (nq < it.nblocks) {
            const uint32_t kbi = kb0 + nq;
            const uint32_t s = kbi % kStages, sb = sc & 1;
            if (mbar_test_wait(&bars[B_KV_FULL0 + s], (kbi / kStages) & 1) &&
                mbar_test_wait(&bars[B_S_EMPTY0 + sb], ((sc >> 1) & 1) ^ 1)) {
              tc_fence_after();
              const uint32_t stg = kvbase + s * kKVStage;
              const uint32_t d = tmem + kTmemS + 64 * sb;
#pragma unroll
              for (int k = 0; k < 16; ++k)  // latent dims 16k.. from TMEM, keys' 64-dim chunk k/4
                mma_bf16_ts(d, tmem + kTmemQ + 8 * k,
                            smem_desc(stg + (k >> 2) * kKVLat + 32 * (k & 3), 16, 1024, kSwizzle128B),
                            idesc_qk, k != 0);
#pragma unroll
              for (int t = 0; t < 2; ++t)
                mma_bf16_ss(d, smem_desc(qrope + 32 * t, 16, 512, kSwizzle64B),
                            smem_desc(stg + 4 * kKVLat + 32 * t, 16, 512, kSwizzle64B), idesc_qk, 1);
              mma_commit(&bars[B_S_FULL0 + sb]);
              ++sc;
              if (++nq == it.nblocks) mma_commit(&bars[B_Q_EMPTY]);  // last use of Q
              did = true;
            }
          }
          if (np < nq) {
            if (!ofree) ofree = mbar_test_wait(&bars[B_O_FREE], (ii & 1) ^ 1);
            if (ofree && mbar_test_wait(&bars[B_P_FULL], pc & 1)) {
              tc_fence_after();
              const uint32_t s = (kb0 + np) % kStages;
              const uint32_t stg = kvbase + s * kKVStage;
#pragma unroll
              for (int t = 0; t < BN / 16; ++t)
                mma_bf16_ts(tmem + kTmemO, tmem + tmem_p_col(t),
                            smem_desc(stg + t * 2048, kKVLat, 1024, kSwizzle128B), idesc_pv,
                            (np | t) != 0);
              mma_commit(&bars[B_KV_EMPTY0 + s]);
              mma_commit(&bars[B_O_DONE]);
              ++pc;
              ++np;
              did = true;
            }
          }
          if (did) {
            idle_since = 0;
          } else {  // nothing ready: bounded like every other wait
            if (*abort) break;
            const long long now = clock64();
            if (idle_since == 0) idle_since = now;
            else if (now - idle_since > kIdleLimitCycles) {
              *abort = 1;
              break;
            }
          }
        }
        kb += it.nblocks;
        ++ii;
      }
      mma_commit(&bars[B_DRAIN]);  // everything issued has completed before TMEM is freed
      mbar_drain(&bars[B_DRAIN], 0, kDrainNs);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ score senders
    // Thread r owns row r (TMEM lane r). As soon as the scores of a block are
    // in TMEM it reads its row of this CTA's partial S_c = Q_c K_c^T, scales
    // it into the log2 domain, rounds it to fp16 and writes it twice: into
    // the own buffer XO and, by st.async, into the peer's buffer XP, whose
    // arrival completes the peer's X_FULL. Both CTAs then form
    // fp32(XO) + fp32(XP) with the same two fp16 terms, so they hold the
    // same scores bit for bit. Working ahead of the softmax warps, the
    // senders overlap a block's exchange with the previous block's softmax.
    const int r = tid - 128;
    const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
    const float scale2 = a.sm_scale * kLog2e;
    const uint32_t xp_peer0 = mapa(smem_u32(sm + kX + kXBytes + r * kXRow), peer);
    const uint32_t xfull_peer0 = mapa(smem_u32(&bars[B_X_FULL0]), peer);
    uint32_t g = 0, qi = 0;
    const int64_t q_rows = (int64_t)a.total_q * H;
    cluster_wait();  // the peer's barriers are initialised
    for (int rnd = 0, id = item_of(0, cluster_id, p.nclusters); id < total_items;
         id = item_of(++rnd, cluster_id, p.nclusters)) {
      const Item it = decode_item(plan, ord, obase, a.batch, id);
      {
        // Row r of the query tile, this CTA's 256 latent dims, into TMEM as
        // bf16 pairs (QK's A operand) once the previous item's last QK is done.
        // Rows past the last query row read as zeros.
        const int64_t qrow = (int64_t)it.q0 * H + it.row0 + r;
        const uint4* src = reinterpret_cast<const uint4*>(a.q + qrow * kDqk + 256 * cta);
        const bool in = qrow < q_rows;
        mbar_wait<false>(&bars[B_Q_EMPTY], (qi & 1) ^ 1, abort);
        ++qi;
        tc_fence_after();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint4 v[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) v[k] = in ? __ldg(src + 16 * half + k) : make_uint4(0, 0, 0, 0);
          uint32_t w0[32], w1[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            w0[4 * k] = v[k].x; w0[4 * k + 1] = v[k].y; w0[4 * k + 2] = v[k].z; w0[4 * k + 3] = v[k].w;
            w1[4 * k] = v[8 + k].x; w1[4 * k + 1] = v[8 + k].y;
            w1[4 * k + 2] = v[8 + k].z; w1[4 * k + 3] = v[8 + k].w;
          }
          tmem_st32(tmem + lane_base + kTmemQ + 64 * half, w0);
          tmem_st32(tmem + lane_base + kTmemQ + 64 * half + 32, w1);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[B_QT_FULL]);
      }
      // kWarm: the first item starts with a dry pass (blk = -1) as in the
      // softmax warps: its waits and signals go to B_DRY, it reads O's
      // columns (not written before the first P.V), writes only the own
      // exchange buffer (rewritten before the softmax may read it) and
      // sends nothing.
      const int warm = (kWarm && rnd == 0) ? 1 : 0;
      g -= warm;
      for (int blk = -warm; blk < it.nblocks; ++blk, ++g) {
        const bool dry = kWarm && blk < 0;
        const uint32_t b = g & 1;
        mbar_wait<false>(&bars[dry ? B_DRY : B_S_FULL0 + b], (g >> 1) & 1, abort);
        tc_fence_after();
        uint32_t s0[32], s1[16];
        const uint32_t tsrc = tmem + lane_base + (dry ? kTmemO : kTmemS + 64 * b);
        tmem_ld32(tsrc, s0);
        tmem_ld16(tsrc + 32, s1);
        tc_fence_before();
        mbar_arrive(&bars[dry ? B_DRY : B_S_EMPTY0 + b]);  // the score buffer may take block g+2
        uint32_t h[BN / 2];
#pragma unroll
        for (int c = 0; c < BN / 2; ++c) {
          const uint32_t u0 = c < 16 ? s0[2 * c] : s1[2 * c - 32];
          const uint32_t u1 = c < 16 ? s0[2 * c + 1] : s1[2 * c - 31];
          // clamp to the finite fp16 range (scores that large saturate the
          // softmax either way)
          const float x0 = fminf(fmaxf(__uint_as_float(u0) * scale2, -65504.f), 65504.f);
          const float x1 = fminf(fmaxf(__uint_as_float(u1) * scale2, -65504.f), 65504.f);
          const __half2 v = __floats2half2_rn(x0, x1);
          h[c] = *reinterpret_cast<const uint32_t*>(&v);
        }
        // both halves of buffer pair b are free: our softmax rows and the
        // peer's have read block g-2
        mbar_wait<true>(&bars[dry ? B_DRY : B_X_FREE0 + b], (((g >> 1) & 1) ^ 1) | (dry ? 1u : 0u), abort);
        uint8_t* xo = sm + kX + 2 * b * kXBytes + r * kXRow;
        const uint32_t dst = xp_peer0 + 2 * b * kXBytes;
        const uint32_t bar = xfull_peer0 + 8 * b;
#pragma unroll
        for (int q = 0; q < BN / 8; ++q) {
          *reinterpret_cast<uint4*>(xo + 16 * q) = make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
          if (!dry) st_async_v4(dst + 16 * q, h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3], bar);
        }
        // own row written; r == 0 also arms the barrier for the peer's bytes
        uint64_t* xfull = &bars[dry ? B_DRY : B_X_FULL0 + b];
        if (r == 0) mbar_arrive_expect_tx(xfull, (uint32_t)(BM * BN * 2));
        else mbar_arrive(xfull);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax, epilogue
    // Block g's scores come from buffer pair g & 1 (XO: ours, XP: the
    // peer's), two pairs so the senders may fill block g+1 while the rows
    // are still on block g.
    const int r = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t t_o = tmem + lane_base + kTmemO;
    const uint32_t xfree_peer0 = mapa(smem_u32(&bars[B_X_FREE0]), peer);
    const int64_t R = (int64_t)a.total_q * H;
    uint32_t pw = 0, gblk = 0;
    cluster_wait();  // the peer's barriers are initialised

    // Give this warp's rows of buffer pair g & 1 back: to our own senders
    // (XO) and to the peer's (our XP is theirs to fill); the pair is free
    // once all four warps of both CTAs have signalled. The rows' reads are
    // complete here (their values were consumed before the signal), so the
    // remote signal needs no release fence.
    auto release_x = [&](uint32_t g) {
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[B_X_FREE0 + (g & 1)]);
        mbar_arrive_remote_relaxed(xfree_peer0 + 8 * (g & 1));
      }
    };

    for (int rnd = 0, id = item_of(0, cluster_id, p.nclusters); id < total_items;
         id = item_of(++rnd, cluster_id, p.nclusters)) {
      const Item it = decode_item(plan, ord, obase, a.batch, id);
      const int rows_req = it.n * H;
      const int row = it.row0 + r;
      const bool valid = row < rows_req;
      const int i_lo = it.row0 / H;
      const int i_hi = min(it.n - 1, (it.row0 + BM - 1) / H);
      const int cnt = i_hi - i_lo + 1;
      const int node = (valid ? row : rows_req - 1) / H;
      // Mask bytes of a block arrive as (draft node, 8-column group) pairs;
      // thread r owns pairs r + 128 k. When a tile touches few enough nodes
      // (every case with 8 or more heads), the bytes of block blk+1 are
      // loaded while block blk is processed.
      const int pre = kSkip ? it.L - it.n : 0;  // prefix columns: visible, mask unread
      constexpr int kGroups = BN / 8;  // 8-column groups per block row
      const int pairs = cnt * kGroups;
      const bool prefetch = pairs <= 128 * kMaskPrefetch;
      uint8_t raw[kMaskPrefetch][8];
      auto load_mask = [&](int blk_) {
        const int jb_ = it.j0 + blk_ * BN;
#pragma unroll
        for (int k = 0; k < kMaskPrefetch; ++k) {
          const int q = r + 128 * k;
          if (q < pairs) {
            const int pos0 = jb_ + 8 * (q % kGroups);
            const uint8_t* src = a.mask + it.mask0 + (int64_t)(i_lo + q / kGroups) * it.L + pos0;
#pragma unroll
            for (int e = 0; e < 8; ++e)
              raw[k][e] = pos0 + e < it.j1 && (!kSkip || pos0 + e >= pre) ? __ldg(src + e) : 0;
          }
        }
      };
      // Bit-form mask: this row's node reads the (up to) three words holding
      // a block's 48 columns straight from global memory, one block ahead.
      const int mw = (it.L + 31) >> 5;
      const uint32_t* mrow = kBits ? a.mask_bits + it.mask0 + (int64_t)node * mw : nullptr;
      uint32_t mnext[3] = {0u, 0u, 0u};
      auto load_bits = [&](int blk_) {
        const int wi = (it.j0 + blk_ * BN) >> 5;
#pragma unroll
        for (int k = 0; k < 3; ++k)
          mnext[k] = wi + k < mw && (!kSkip || 32 * (wi + k) + 32 > pre) ? __ldg(mrow + wi + k) : 0u;
      };
      if (kBits) load_bits(0);
      else if (prefetch) load_mask(0);
      float m = -INFINITY, l = 0.f;
      // kWarm: the first item starts with a dry pass (blk = -1) over the
      // block body while the first scores are still in flight, only to pull
      // the body's instructions into the SM's caches ahead of the real first
      // block. It waits on and signals B_DRY (its wait parity, from a
      // counter one below the first block's, is that of a phase counted as
      // complete), releases nothing, and its P store lands in columns no
      // MMA reads yet.
      const int warm = (kWarm && rnd == 0) ? 1 : 0;
      gblk -= warm;
      for (int blk = -warm; blk < it.nblocks; ++blk, ++gblk) {
        const bool dry = kWarm && blk < 0;
        const int jb = it.j0 + blk * BN;
        uint64_t vm;
        if (kBits) {
          const uint32_t w0 = mnext[0], w1 = mnext[1], w2 = mnext[2];
          if (blk + 1 < it.nblocks) load_bits(blk + 1);
          const int o = jb & 31;
          const uint64_t lo = (uint64_t)w0 | ((uint64_t)w1 << 32);
          vm = o ? (lo >> o) | ((uint64_t)w2 << (64 - o)) : lo;
          const int lim = it.j1 - jb;  // columns of this block inside the split
          if (lim < 64) vm &= (1ull << lim) - 1ull;
        } else {
        // visibility bits of this block for the tile's draft nodes
        uint8_t* vb = reinterpret_cast<uint8_t*>(vis + (gblk & 1) * kVisNodes);
        if (prefetch) {
#pragma unroll
          for (int k = 0; k < kMaskPrefetch; ++k) {
            const int q = r + 128 * k;
            if (q < pairs) {
              uint32_t bits = 0;
#pragma unroll
              for (int e = 0; e < 8; ++e) bits |= (raw[k][e] != 0 ? 1u : 0u) << e;
              vb[(q / kGroups) * 8 + q % kGroups] = (uint8_t)bits;
            }
          }
          if (blk + 1 < it.nblocks) load_mask(blk + 1);
        } else {
          for (int q = r; q < pairs; q += 128) {
            const int pos0 = jb + 8 * (q % kGroups);
            const uint8_t* src = a.mask + it.mask0 + (int64_t)(i_lo + q / kGroups) * it.L + pos0;
            uint32_t bits = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (pos0 + e < it.j1 && (!kSkip || pos0 + e >= pre) && __ldg(src + e)) bits |= 1u << e;
            vb[(q / kGroups) * 8 + q % kGroups] = (uint8_t)bits;
          }
        }
        named_bar_sync(1, 128);
        vm = vis[(gblk & 1) * kVisNodes + (node - i_lo)];
        }
        if (kSkip && pre > jb) {  // the block's prefix columns, up to the split's end
          const int pc = min(pre, it.j1) - jb;
          vm |= pc >= 64 ? ~0ull : (1ull << pc) - 1ull;
        }

        // full scores (log2 domain): our fp16 partial plus the peer's
        const uint32_t xb = gblk & 1;
        mbar_wait<true>(&bars[dry ? B_DRY : B_X_FULL0 + xb], (gblk >> 1) & 1, abort);
        const uint8_t* xo = sm + kX + 2 * xb * kXBytes + r * kXRow;
        const uint8_t* xp = xo + kXBytes;
        float s[BN];
#pragma unroll
        for (int q = 0; q < BN / 8; ++q) {
          const uint4 u = *reinterpret_cast<const uint4*>(xo + 16 * q);
          const uint4 v = *reinterpret_cast<const uint4*>(xp + 16 * q);
          const uint32_t uu[4] = {u.x, u.y, u.z, u.w}, vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 fu = __half22float2(*reinterpret_cast<const __half2*>(&uu[e]));
            const float2 fv = __half22float2(*reinterpret_cast<const __half2*>(&vv[e]));
            s[8 * q + 2 * e] = fu.x + fv.x;
            s[8 * q + 2 * e + 1] = fu.y + fv.y;
          }
        }
        // the last block's pair stays ours: the epilogue stages rows in it
        if (kWarm ? (unsigned)blk < (unsigned)(it.nblocks - 1) : blk + 1 < it.nblocks) release_x(gblk);

        // masked online softmax (log2 domain)
        const uint32_t vlo = (uint32_t)vm, vhi = (uint32_t)(vm >> 32);
        float mx[8];  // eight independent running maxima, then a tree
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const uint32_t bit = c < 32 ? (vlo >> c) & 1u : (vhi >> (c - 32)) & 1u;
          const float v = bit ? s[c] : -INFINITY;
          s[c] = v;
          mx[c & 7] = c < 8 ? v : fmaxf(mx[c & 7], v);
        }
        const float mb = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        float corr = 1.f;
        bool resc = false;
        if (mb > m + kRescale) {
          corr = ex2_approx(m - mb);
          m = mb;
          resc = true;
        }
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[BN / 2];
        if (m == -INFINITY) {
#pragma unroll
          for (int c = 0; c < BN / 2; ++c) pk[c] = 0u;
        } else {
#pragma unroll
          for (int c = 0; c < BN / 2; ++c) {
            const float p0 = ex2_approx(s[2 * c] - m), p1 = ex2_approx(s[2 * c + 1] - m);
            const __nv_bfloat162 v = __floats2bfloat162_rn(p0, p1);
            // the denominator sums the same bf16 weights the P.V product uses,
            // so O / l stays a true weighted average of the value rows
            rs4[c & 3] += __low2float(v) + __high2float(v);
            pk[c] = *reinterpret_cast<const uint32_t*>(&v);
          }
        }
        l = l * corr + ((rs4[0] + rs4[1]) + (rs4[2] + rs4[3]));

        // the previous P.V is done: P and O may be touched
        if (blk > 0) {
          mbar_wait<false>(&bars[B_O_DONE], pw & 1, abort);
          ++pw;
          tc_fence_after();
        }
        const bool need = resc && blk > 0;
        if (__any_sync(0xffffffffu, need)) {
          const float f = need ? corr : 1.f;
#pragma unroll 1
          for (int k = 0; k < 8; ++k) {
            uint32_t o[32];
            tmem_ld32(t_o + 32 * k, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32(t_o + 32 * k, o);
          }
        }
        {  // row r of P: 48 bf16 weights as 24 packed columns, in two pieces
          uint32_t p01[16], p2[8];
#pragma unroll
          for (int c = 0; c < 16; ++c) p01[c] = pk[c];
#pragma unroll
          for (int c = 0; c < 8; ++c) p2[c] = pk[16 + c];
          tmem_st16(tmem + lane_base + tmem_p_col(0), p01);
          tmem_st8(tmem + lane_base + tmem_p_col(2), p2);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[dry ? B_DRY : B_P_FULL]);
        if (dry) {
          m = -INFINITY;
          l = 0.f;
        }
      }
      const uint32_t glast = gblk - 1;

      // epilogue: O / l for this CTA's 256 value dims. Each 128-byte piece of
      // every row goes through the last block's exchange buffer (still held),
      // so a warp stores four whole 128-byte row pieces per instruction
      // instead of 32 scattered 16-byte pieces.
      mbar_wait<false>(&bars[B_O_DONE], pw & 1, abort);
      ++pw;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t row_base = (int64_t)it.q0 * H + it.row0;
      const int valid_rows = min(BM, rows_req - it.row0);
      uint8_t* stage = sm + kX + 2 * (glast & 1) * kXBytes;
      named_bar_sync(3, 128);  // every row has read the last block's scores
      if (it.splits == 1) {
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {  // 64 bf16 columns per round
          uint32_t o0[32], o1[32];
          tmem_ld32(t_o + 64 * k, o0);
          tmem_ld32(t_o + 64 * k + 32, o1);
          uint32_t w[32];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const __nv_bfloat162 v0 = __floats2bfloat162_rn(__uint_as_float(o0[2 * e]) * inv,
                                                            __uint_as_float(o0[2 * e + 1]) * inv);
            const __nv_bfloat162 v1 = __floats2bfloat162_rn(__uint_as_float(o1[2 * e]) * inv,
                                                            __uint_as_float(o1[2 * e + 1]) * inv);
            w[e] = *reinterpret_cast<const uint32_t*>(&v0);
            w[16 + e] = *reinterpret_cast<const uint32_t*>(&v1);
          }
#pragma unroll
          for (int g = 0; g < 8; ++g)
            *reinterpret_cast<uint4*>(stage + r * 128 + ((g ^ (r & 7)) << 4)) =
                make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
          named_bar_sync(3, 128);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int idx = i * 128 + r, rl = idx >> 3, g = idx & 7;
            if (rl < valid_rows)
              *reinterpret_cast<uint4*>(a.out + (row_base + rl) * kDv + 256 * cta + 64 * k + 8 * g) =
                  *reinterpret_cast<const uint4*>(stage + rl * 128 + ((g ^ (rl & 7)) << 4));
          }
          named_bar_sync(3, 128);
        }
      } else {
        // split partials in fp16 (each is a convex combination of value rows;
        // 11 significand bits keep it far below the bf16 output rounding)
        __half* wso = reinterpret_cast<__half*>(a.ws_o) + ((int64_t)it.split * R + row_base) * kDv + 256 * cta;
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {  // 64 columns per round
          uint32_t o0[32], o1[32];
          tmem_ld32(t_o + 64 * k, o0);
          tmem_ld32(t_o + 64 * k + 32, o1);
          uint32_t w[32];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const __half2 v0 = __floats2half2_rn(__uint_as_float(o0[2 * e]) * inv,
                                                 __uint_as_float(o0[2 * e + 1]) * inv);
            const __half2 v1 = __floats2half2_rn(__uint_as_float(o1[2 * e]) * inv,
                                                 __uint_as_float(o1[2 * e + 1]) * inv);
            w[e] = *reinterpret_cast<const uint32_t*>(&v0);
            w[16 + e] = *reinterpret_cast<const uint32_t*>(&v1);
          }
#pragma unroll
          for (int g = 0; g < 8; ++g)
            *reinterpret_cast<uint4*>(stage + r * 128 + ((g ^ (r & 7)) << 4)) =
                make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
          named_bar_sync(3, 128);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int idx = i * 128 + r, rl = idx >> 3, g = idx & 7;
            if (rl < valid_rows)
              *reinterpret_cast<uint4*>(wso + (int64_t)rl * kDv + 64 * k + 8 * g) =
                  *reinterpret_cast<const uint4*>(stage + rl * 128 + ((g ^ (rl & 7)) << 4));
          }
          named_bar_sync(3, 128);
        }
      }
      if (valid && cta == 0) {
        const float lv = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        const int64_t grow = row_base + r;
        if (it.splits == 1) a.lse[grow] = lv;
        else a.ws_lse[(int64_t)it.split * R + grow] = lv;
      }
      tc_fence_before();
      mbar_arrive(&bars[B_O_FREE]);  // O has been read: the next item may overwrite it
      release_x(glast);  // staging done: the peer may refill this buffer
    }
  }

  if (warp >= kFirstProducer) cluster_wait();  // pairs with the arrival after set-up
  // this CTA's outputs are issued: the merge kernel (launched as a dependent
  // grid) may start its set-up; it waits for this grid's completion before
  // reading any partial
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0 && *abort) flag(a.status, MT_DEV_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();  // no CTA leaves while its peer may still write into it
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
std::mutex g_dev_mu;
int g_clusters[64] = {0};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// 2-D map over rows of 576 bf16 (1152-byte pitch), box box_cols x box_rows.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows, CUtensorMapSwizzle sw) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kDqk, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kDqk * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

using KernelFn = void (*)(TcParams, CUtensorMap, CUtensorMap, CUtensorMap);

// The instantiations: byte mask (no dry pass) or bit mask, each with and
// without the prefix skip.
constexpr int kVariants = 6;
KernelFn kernel_variant(int i) {
  switch (i) {
    case 0: return verify_tc_kernel<false, false, false>;
    case 1: return verify_tc_kernel<false, false, true>;
    case 2: return verify_tc_kernel<true, false, false>;
    case 3: return verify_tc_kernel<true, false, true>;
    case 4: return verify_tc_kernel<true, true, false>;
    default: return verify_tc_kernel<true, true, true>;
  }
}
int variant_index(bool bits, bool warm, bool skip) {
  return !bits ? (skip ? 1 : 0) : (warm ? 4 : 2) + (skip ? 1 : 0);
}

// Clusters of two that fit at once on this device (persistent grid size).
int device_clusters(int num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (g_clusters[dev] > 0) return g_clusters[dev];
  for (int i = 0; i < kVariants; ++i)
    if (cudaFuncSetAttribute(kernel_variant(i), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (num_sms / 2));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel_variant(0), &cfg) != cudaSuccess || n <= 0)
    n = num_sms / 2;
  g_clusters[dev] = n;
  return n;
}

}  // namespace tc

cudaError_t launch_verify_tc(const VerifyArgs& a, int num_sms, cudaStream_t stream) {
  using namespace tc;
  if (a.batch > kMaxBatch || a.num_slots <= 0 || a.num_slots >= 0x7fffffffLL ||
      (long long)a.total_q * a.heads >= 0x7fffffffLL)
    return cudaErrorNotSupported;
  const int nclusters = device_clusters(num_sms > 0 ? num_sms : 148);
  if (nclusters <= 0) return cudaErrorNotSupported;
  CUtensorMap tq_rope, tkv_lat, tkv_rope;
  const uint64_t qrows = (uint64_t)a.total_q * a.heads;
  if (!make_map(&tq_rope, a.q, qrows, 32, BM, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&tkv_lat, a.kv, (uint64_t)a.num_slots, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&tkv_rope, a.kv, (uint64_t)a.num_slots, 32, 1, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorNotSupported;
  TcParams p;
  p.a = a;
  p.a.partial_f16 = 1;
  p.nclusters = nclusters;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * nclusters);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the previous kernel in the stream finishes (the kernel
  // waits for it before reading anything)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // The dry passes cost a few instructions in every block and save a few
  // microseconds of instruction fetch once per CTA: they pay when each
  // cluster has at most a few hundred key blocks to do. An upper bound from
  // the host-known sizes (every tile against the whole kv_indices) decides.
  const long long tiles_ub = ((long long)a.total_q * a.heads + BM - 1) / BM + a.batch;
  const bool warm = a.bits_mask && tiles_ub * a.kv_len <= (long long)kWarmBlocks * BN * nclusters;
  const KernelFn fn = kernel_variant(variant_index(a.bits_mask != 0, warm, a.skip_prefix != 0));
  cudaError_t e = cudaLaunchKernelEx(&cfg, fn, p, tq_rope, tkv_lat, tkv_rope);
  if (e != cudaSuccess) return e;
  if (a.max_splits > 1) return launch_lse_merge(p.a, stream);
  return cudaSuccess;
}

int verify_tc_launches(int batch, int total_q, int heads, int max_splits) {
  (void)total_q;
  (void)heads;
  if (batch > tc::kMaxBatch) return 0;
  return max_splits > 1 ? 2 : 1;
}

}  // namespace mt
