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
// query tile and of every key row, and a 256-dim half of the output
// accumulator O. The softmax is split by rows instead: CTA c owns tile rows
// [64c, 64c+64). Per block of BN = 48 key rows:
//
//   TMA       key-row halves by tile::gather4 through kv_indices, four rows
//             per instruction, several stages in flight
//   tcgen05   S_c = Q_c K_c^T   (M=128, N=48, K=288) into TMEM
//   DSMEM     each CTA sends its fp32 partial scores of the rows the other
//             CTA owns (64 rows x 48) to that CTA; with the byte-form mask
//             the senders apply the mask (a hidden column is sent as -inf)
//   softmax   the owner adds the two fp32 partials (exact scores of its
//             rows, in the log2 domain), applies the bit-form mask and runs the
//             online softmax (four threads per row, 12 columns each; lazy
//             rescaling: the running max moves only when it grows by more
//             than 8, i.e. a factor of 256); it writes its rows of P (bf16)
//             to its own TMEM and sends them, with the running max and
//             sums, to the other CTA, which writes them into its TMEM (and
//             rescales its half of those rows of O when the max moved)
//   tcgen05   O_c += P V_c      (M=128, N=256, K=48) into TMEM; V_c is the
//             same shared-memory key tile, read MN-major
//
// Why two CTAs: a 128-row fp32 accumulator for all 512 value dims is the
// whole 256 KB of TMEM. Splitting the dims halves it and leaves TMEM room
// for 224 of the query half's 256 latent dims (14 of a block's 18 QK MMAs
// take the query from TMEM; the last 32 latent dims and the rope half come
// from shared memory), two score buffers and two P buffers. The scores cross
// between the CTAs in fp32, so no partial is rounded below fp32 before the
// softmax.
//
// Roles per CTA (512 threads, 16 warps; a warp's TMEM lane quarter and its
// scheduler are warp % 4): in CTA c the eight warps whose quarter holds the
// own rows run the softmax (four threads per row) and the own rows'
// epilogue, so the own rows' two schedulers run nothing else. On the other
// two schedulers, warps 0-3 send partial scores (and apply a byte-form
// mask), warps 4-7 receive P and run those rows' epilogue, and of warps
// 8-15 one issues the MMAs and owns TMEM while three are TMA producers (one
// warp alone issues tile::gather4 too slowly to keep up). Every mbarrier wait is time-bounded: a timeout sets
// MT_DEV_TIMEOUT, after which no thread issues another copy, MMA or remote
// store, every loop runs to its end (so no named barrier is left waiting)
// and the copies and MMAs in flight are drained before TMEM is released.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "mt_common.cuh"
#include "mt_internal.h"
#include "sm100_ptx.cuh"

namespace mt {
namespace tc {

using namespace sm100;

constexpr int BM = 128;          // tile rows = TMEM lanes
constexpr int BN = 48;           // key rows per block
constexpr int kOwnRows = BM / 2; // rows whose softmax a CTA runs
constexpr int kRowThreads = 4;   // softmax threads per own row, in four warps of the row's quarter
constexpr int kQCols = BN / kRowThreads;  // columns per softmax thread
constexpr int kSoftThreads = kOwnRows * kRowThreads;  // 256
constexpr int kGatherLanes = BN / 4;  // four-row groups per block (tile::gather4)
constexpr int kProducers = 3;    // TMA producer warps (one warp issues about 37 ns per gather4)
constexpr int kThreads = 512;    // 16 warps
static_assert(kProducers == 3, "warps 8-15 of the two non-softmax quarters: one MMA issuer, three producers");
constexpr int kMaxBatch = 256;   // requests per launch (the plan lives in shared memory)
constexpr float kRescale = 8.f;  // lazy-rescale threshold (log2 units)
constexpr int kMinChunk = 256;   // smallest split worth a work item (key rows)
constexpr int kMaskPrefetch = 2; // byte-mask (node, group) pairs per score-sender thread held one block ahead
constexpr int kSlotAhead = 2;    // key blocks whose slot numbers are in flight ahead of the gathers
constexpr int kGroupsPerWarp = kGatherLanes / kProducers;
static_assert(kGatherLanes % kProducers == 0, "groups per producer warp");

// Shared memory map (offsets from a 1024-byte aligned base).
constexpr int kQRope = 0;                             // query rope half [128 rows x 64 B], 64B swizzle
constexpr int kQTail = kQRope + BM * 64;              // query latent dims 224..255 of the CTA's half, same form
constexpr int kKV = kQTail + BM * 64;                 // key stages
constexpr int kKVLat = BN * 128;                      // one latent chunk of a stage
constexpr int kKVStage = 4 * kKVLat + BN * 64;        // 27648
constexpr int kStages = 5;
constexpr int kSX = kKV + kStages * kKVStage;         // the peer's fp32 partial scores of our rows, 2 buffers
// The exchange buffers are chunk-major: 16-byte chunk k of row r sits at
// k * kXChunk + 16 r, so the 32 remote stores of one warp instruction (32
// rows, one chunk each) fill 512 contiguous bytes, whole 32-byte sectors.
constexpr int kXChunk = kOwnRows * 16;
constexpr int kSXChunks = BN * 4 / 16;                // 12 chunks of 4 fp32 partial scores
constexpr int kSXBytes = kSXChunks * kXChunk;
constexpr int kPX = kSX + 2 * kSXBytes;               // the peer's P rows (+ running max, sums), 2 buffers
// P rows go in 8-byte chunks (a softmax thread's 12 keys are 24 bytes): chunk
// k of row r at k * kPChunk + 8 r; chunks 0..11 hold P, chunk 12 + h holds
// (m, l_h) of the row's thread h
constexpr int kPChunk = kOwnRows * 8;
constexpr int kPXChunks = BN * 2 / 8 + kRowThreads;   // 16
constexpr int kPXBytes = kPXChunks * kPChunk;
constexpr int kMX = kPX + 2 * kPXBytes;               // quarter-row maxima [2][64][4] and sums [64][4]
constexpr int kVisNodes = BM + 2;                     // distinct draft nodes a tile can touch
constexpr int kVis = kMX + (2 * kOwnRows * kRowThreads + kOwnRows * kRowThreads) * 4;  // 2 x kVisNodes x 64-bit masks
constexpr int kBars = kVis + 2 * kVisNodes * 8;
constexpr int B_Q_FULL = 0;                     // query rope half landed (TMA)
constexpr int B_QT_FULL = 1;                    // query latent half written to TMEM
constexpr int B_Q_EMPTY = 2;                    // last QK of the item done
constexpr int B_KV_FULL0 = 3;                   // kStages x kProducers: one per producer warp
constexpr int B_KV_EMPTY0 = B_KV_FULL0 + kStages * kProducers;
constexpr int B_S_FULL0 = B_KV_EMPTY0 + kStages;  // two each from here
constexpr int B_S_EMPTY0 = B_S_FULL0 + 2;
constexpr int B_SX_FULL0 = B_S_EMPTY0 + 2;
constexpr int B_SX_FREE0 = B_SX_FULL0 + 2;
constexpr int B_PX_FULL0 = B_SX_FREE0 + 2;
constexpr int B_PX_FREE0 = B_PX_FULL0 + 2;
constexpr int B_P_FULL0 = B_PX_FREE0 + 2;        // one per P buffer
constexpr int B_O_DONE0 = B_P_FULL0 + 2;        // P.V done, one per P buffer it read
constexpr int B_O_FREE = B_O_DONE0 + 2;
constexpr int B_DRAIN = B_O_FREE + 1;
constexpr int kNumBars = B_DRAIN + 1;
constexpr int kMisc = kBars + kNumBars * 8;           // tmem base, abort flag, item count, wait limit
constexpr int kPlan = kMisc + 32;                     // per-request plan
constexpr int kPlanStride = 9;                        // int32 words per request
constexpr int kOrd = kPlan + kMaxBatch * kPlanStride * 4;   // request at each rank
constexpr int kOBase = kOrd + kMaxBatch * 4;          // first item of each rank (+ total)
constexpr int kSmemUsed = kOBase + (kMaxBatch + 1) * 4;
constexpr int kSmemBytes = kSmemUsed + 1024;          // slack for aligning the base
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(BN % 16 == 0 && BN <= 64, "block width");
static_assert(kQRope % 1024 == 0 && kQTail % 1024 == 0 && kKV % 1024 == 0 && kKVStage % 1024 == 0 && kSX % 16 == 0 &&
                  kPX % 16 == 0 && kBars % 8 == 0 &&
                  kMisc % 8 == 0,
              "alignment");

constexpr uint32_t kQTx = 2 * BM * 64;                // query rope + latent-tail bytes per CTA per item
constexpr uint32_t kKVTxWarp = kGroupsPerWarp * 4 * (4 * 128 + 64);  // key bytes per producer warp per block
constexpr uint32_t kSXTx = kOwnRows * BN * 4;         // partial-score bytes into a CTA per block
constexpr uint32_t kPXTx = kPXBytes;                  // P + (m, l_h) bytes into a CTA per block
static_assert(kKVTxWarp * kProducers == (uint32_t)kKVStage, "stage bytes");
constexpr uint32_t kTmemCols = 512;
// TMEM columns (512 x 128 lanes; lane = tile row):
//   [0, 256)    O, this CTA's 256 value dims (fp32)
//   [256, 368)  Q, latent dims 0..223 of this CTA's half as bf16 pairs: QK's
//               A operand for 14 of its 16 K steps (dims 224..255 and the
//               rope come from shared memory)
//   [384, 432)  S buffer 0, [448, 496) S buffer 1 (BN fp32 scores each)
//   P (bf16 pairs, PV's A), two buffers, one 8-column piece per 16 keys:
//   buffer 0 at [432, 448) and [496, 504), buffer 1 at [368, 384) and
//   [504, 512). Two P buffers let P of block g+1 be written while the
//   P.V of block g still reads P of block g.
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemQ = 256;
constexpr int kQTmemSteps = 14;                       // QK K steps with A in TMEM
constexpr uint32_t kTmemS = 384;                      // buffer b at kTmemS + 64 b
__host__ __device__ constexpr uint32_t tmem_p_col(int pb, int t) {
  return pb == 0 ? (t < 2 ? 432u + 8u * t : 496u) : (t < 2 ? 368u + 8u * t : 504u);
}
static_assert(BN == 48, "TMEM map holds 48-column score blocks and three P pieces");
static_assert(kTmemQ + 8 * kQTmemSteps == 368, "Q ends where P buffer 1 starts");
constexpr uint64_t kDrainNs = 100000000ull;           // 100 ms
constexpr uint64_t kAbortSettleNs = 50000ull;         // after a give-up: let remote stores land

// plan words
enum { PL_Q0, PL_N, PL_KV0, PL_L, PL_SPLITS, PL_LEN, PL_TILES, PL_M0LO, PL_M0HI };

// Optional pipeline trace for studying the kernel (off unless the library
// is compiled with -DMT_TC_TRACE): %globaltimer at fixed points of the first
// kTrBlocks key blocks of the first cluster's two CTAs, one thread per role,
// in g_tc_trace[cta][role][block][event]; read with mla_tree_tc_trace_read.
// Events 3-9 of the receiver role at block 0 mark the kernel's phases
// (TC_MARK): entry, grid dependency resolved, plan ready, softmax and
// receiver epilogues done, exit.
enum { TR_PRODUCER, TR_MMA, TR_SENDER, TR_SOFTMAX, TR_RECEIVER, kTrRoles };
#ifdef MT_TC_TRACE
constexpr int kTrCtas = 2, kTrBlocks = 1024, kTrEvents = 10;
__device__ unsigned long long g_tc_trace[kTrCtas][kTrRoles][kTrBlocks][kTrEvents];
#define TC_TRACE(on, role, blk, ev)                                              \
  do {                                                                           \
    if ((on) && blockIdx.x < kTrCtas && (unsigned)(blk) < (unsigned)kTrBlocks)   \
      g_tc_trace[blockIdx.x][role][blk][ev] = global_timer_ns();                 \
  } while (0)
#define TC_MARK(on, ev) TC_TRACE(on, TR_RECEIVER, 0, ev)
#else
#define TC_MARK(on, ev) \
  do {                  \
  } while (0)
#define TC_TRACE(on, role, blk, ev) \
  do {                              \
  } while (0)
#endif

struct TcParams {
  VerifyArgs a;          // one chunk of at most kMaxBatch requests (indptrs offset to it)
  int nclusters;
  int first_chunk;       // the chunk holding request 0 / the last request: bounds of the
  int last_chunk;        //   token range whose split counts this launch publishes
  int drop_item;         // test hook: producers issue nothing from this item on (-1: off)
  unsigned long long limit_ns;  // bound of every wait
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
__device__ void build_plan(const TcParams& p, int* plan, int* ord, int* obase, int* total_items,
                           int lane, bool publish) {
  const VerifyArgs& a = p.a;
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
  const long long nc = p.nclusters > 0 ? p.nclusters : 1;
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
  // tokens of this launch's range that no consistent request covers (an
  // inconsistent request, or outside every request) are not merged
  if (publish) {
    __syncwarp();
    int tlo = p.first_chunk ? 0 : a.qo_indptr[0];
    int thi = p.last_chunk ? a.total_q : a.qo_indptr[a.batch];
    tlo = max(0, tlo);
    thi = min(a.total_q, thi);
    for (int tk = tlo + lane; tk < thi; tk += 32) {
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

// A softmax thread's 28 query columns into TMEM as three naturally aligned
// pieces: 16 columns at O16, 8 at O8, 4 at O4 (offsets within the 28).
template <int O16, int O8, int O4>
__device__ __forceinline__ void tmem_st_q28(uint32_t tq, const uint32_t (&w)[28]) {
  uint32_t a16[16], a8[8], a4[4];
#pragma unroll
  for (int k = 0; k < 16; ++k) a16[k] = w[O16 + k];
#pragma unroll
  for (int k = 0; k < 8; ++k) a8[k] = w[O8 + k];
#pragma unroll
  for (int k = 0; k < 4; ++k) a4[k] = w[O4 + k];
  tmem_st16(tq + O16, a16);
  tmem_st8(tq + O8, a8);
  tmem_st4(tq + O4, a4);
}

// kBits: the tree mask is in the bit form (rows of ceil(L / 32) words)
// kSkip: prefix columns are visible and their mask entries are not read
template <bool kBits, bool kSkip>
__global__ void __launch_bounds__(kThreads, 1)
    verify_tc_kernel(const __grid_constant__ TcParams p,
                     const __grid_constant__ CUtensorMap tm_qrope,
                     const __grid_constant__ CUtensorMap tm_kvlat,
                     const __grid_constant__ CUtensorMap tm_kvrope) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const VerifyArgs& a = p.a;
  const int H = a.heads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t cta = cluster_ctarank();
  const uint32_t peer = cta ^ 1u;
  // Warps 8-15 on the two schedulers that run no softmax warp (CTA 0's own
  // rows are lane quarters 0-1, CTA 1's quarters 2-3): the first issues the
  // MMAs, the other three produce.
  const int mma_warp = cta ? 8 : 10;
  const int cluster_id = blockIdx.x >> 1;
  const uint64_t limit = p.limit_ns;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + kMisc + 4);
  int* total_items_s = reinterpret_cast<int*>(sm + kMisc + 8);
  int* plan = reinterpret_cast<int*>(sm + kPlan);
  int* ord = reinterpret_cast<int*>(sm + kOrd);
  int* obase = reinterpret_cast<int*>(sm + kOBase);
  uint64_t* vis = reinterpret_cast<uint64_t*>(sm + kVis);
  float* mxs = reinterpret_cast<float*>(sm + kMX);               // [2][64][4] quarter-row maxima
  float* lxs = mxs + 2 * kOwnRows * kRowThreads;                 // [64][4] quarter-row sums

  if (tid == 0) {
    mbar_init(&bars[B_Q_FULL], 1);
    mbar_init(&bars[B_QT_FULL], kSoftThreads / 32 + 2);  // softmax and sender warps
    mbar_init(&bars[B_Q_EMPTY], 1);
    for (int s = 0; s < kStages; ++s) {
      for (int w = 0; w < kProducers; ++w) mbar_init(&bars[B_KV_FULL0 + s * kProducers + w], 1);
      mbar_init(&bars[B_KV_EMPTY0 + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[B_S_FULL0 + s], 1);
      mbar_init(&bars[B_S_EMPTY0 + s], kSoftThreads / 32 + 2);  // softmax and sender warps
      mbar_init(&bars[B_SX_FULL0 + s], 1);            // armed once per block, + the peer's bytes
      mbar_init(&bars[B_SX_FREE0 + s], kSoftThreads / 32);  // the peer's softmax warps
      mbar_init(&bars[B_PX_FULL0 + s], 1);
      mbar_init(&bars[B_PX_FREE0 + s], 2);            // the peer's two receiver warps
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[B_P_FULL0 + s], kSoftThreads / 32 + 2);  // softmax and receiver warps
      mbar_init(&bars[B_O_DONE0 + s], 1);
    }
    mbar_init(&bars[B_O_FREE], kSoftThreads / 32 + 2);  // softmax and receiver warps
    mbar_init(&bars[B_DRAIN], 1);
    *abort = 0;
    fence_mbar_init_cluster();
    // the first two blocks' exchange buffers are expected before any
    // arrival from the peer is possible (the peer waits for the cluster
    // barrier below)
    for (int s = 0; s < 2; ++s) {
      mbar_arrive_expect_tx(&bars[B_SX_FULL0 + s], kSXTx);
      mbar_arrive_expect_tx(&bars[B_PX_FULL0 + s], kPXTx);
    }
  }
  if (warp == mma_warp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 9 && lane == 0) {
    prefetch_tmap(&tm_qrope);
    prefetch_tmap(&tm_kvlat);
    prefetch_tmap(&tm_kvrope);
  }
  // Launched as a programmatic dependent of the kernel before it (the
  // marshaling of the same step): the set-up above overlaps that kernel's
  // tail; nothing it writes is read before it has completed.
  TC_MARK(tid == 0, 3);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  TC_MARK(tid == 0, 4);
  // the last CTA publishes the split counts: with fewer items than clusters it
  // has none of its own, so the extra stores delay no item
  if (warp == 0) build_plan(p, plan, ord, obase, total_items_s, lane, blockIdx.x == gridDim.x - 1);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  TC_MARK(tid == 0, 5);
  // The peer's barriers must exist before anyone touches them remotely: every
  // thread arrives here, and the warps that reach into the peer wait before
  // their first remote access; the others wait at the end.
  cluster_arrive();
  const uint32_t tmem = *tmem_slot;
  const int total_items = *total_items_s;
  const int q4 = warp & 3;                       // TMEM lane quarter of this warp
  const bool own_quarter = (uint32_t)(q4 >> 1) == cta;
  const int wg = warp >> 2;
  const bool is_mma = warp == mma_warp;
  const bool is_producer = !own_quarter && wg >= 2 && !is_mma;
  const int64_t q_rows = (int64_t)a.total_q * H;
  const int64_t R = q_rows;

  if (is_producer) {
    // ------------------------------------------------------------ producers
    // kProducers warps share every block's gathers: warp pw issues the
    // four-row groups [pw * kGroupsPerWarp, (pw + 1) * kGroupsPerWarp), one
    // group per lane, and completes its own barrier of the stage (so it can
    // drain exactly the copies it issued). The first producer warp also
    // loads the query tile's rope half.
    const int pw = (wg - 2) * 2 + (q4 & 1) - 1;  // the MMA issuer is the first of the four
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
    bool stop = false;
    for (int rnd = 0, id = item_of(0, cluster_id, p.nclusters); id < total_items && !stop;
         id = item_of(++rnd, cluster_id, p.nclusters)) {
      if (id == p.drop_item) break;  // test hook: the waits on this item's keys must give up
      const Item it = decode_item(plan, ord, obase, a.batch, id);
      const int qrow = it.q0 * H + it.row0;
      if (pw == 0) {
        int ok = 0;
        if (lane == 0 && mbar_wait<false>(&bars[B_Q_EMPTY], (qi & 1) ^ 1, abort, limit) && !*abort) {
          mbar_arrive_expect_tx(&bars[B_Q_FULL], kQTx);
          tma_load_2d(sm + kQRope, &tm_qrope, 512 + 32 * (int)cta, qrow, &bars[B_Q_FULL]);
          tma_load_2d(sm + kQTail, &tm_qrope, 256 * (int)cta + 224, qrow, &bars[B_Q_FULL]);
          ok = 1;
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;  // given up: issue nothing more
        ++qi;
      }
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
      for (int blk0 = 0; blk0 < it.nblocks && !stop; blk0 += kSlotAhead) {
#pragma unroll
        for (int u = 0; u < kSlotAhead; ++u) {
          const int blk = blk0 + u;
          if (blk < it.nblocks && !stop) {
            const int s = kb % kStages;
            uint8_t* st = sm + kKV + s * kKVStage;
            uint64_t* full = &bars[B_KV_FULL0 + s * kProducers + pw];
            int go = 0;
            if (lane == 0) {
              go = mbar_wait<false>(&bars[B_KV_EMPTY0 + s], ((kb / kStages) & 1) ^ 1, abort, limit) &&
                   !*abort;
              if (go) mbar_arrive_expect_tx(full, kKVTxWarp);
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            TC_TRACE(pw == 0 && lane == 0, TR_PRODUCER, kb, 0);
            if (!go) {  // given up: issue nothing more
              stop = true;
              break;
            }
            if (gathers) {
              int rows[4];
              take_rows(ring[u], live[u], rows);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                tma_gather4(st + k * kKVLat + grp * 512, &tm_kvlat, 256 * (int)cta + 64 * k,
                            rows[0], rows[1], rows[2], rows[3], full);
              tma_gather4(st + 4 * kKVLat + grp * 256, &tm_kvrope, 512 + 32 * (int)cta, rows[0],
                          rows[1], rows[2], rows[3], full);
              live[u] = 0;
              if (blk + kSlotAhead < it.nblocks) load_rows(it, blk + kSlotAhead, ring[u], live[u]);
            }
            __syncwarp();
            TC_TRACE(pw == 0 && lane == 0, TR_PRODUCER, kb, 1);
            ++kb;
          }
        }
      }
    }
    if (lane == 0) {  // every copy this warp issued has landed before the CTA may exit
      if (pw == 0 && qi > 0) mbar_drain(&bars[B_Q_FULL], (qi - 1) & 1, kDrainNs);
      for (uint32_t k = kb >= kStages ? kb - kStages : 0; k < kb; ++k)
        mbar_drain(&bars[B_KV_FULL0 + (k % kStages) * kProducers + pw], (k / kStages) & 1, kDrainNs);
    }
  } else if (is_mma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t kb = 0, sc = 0, pc = 0, qi = 0, ii = 0;
      const uint32_t idesc_qk = idesc_bf16(BM, BN, 0, 0);
      const uint32_t idesc_pv = idesc_bf16(BM, 256, 0, 1);
      const uint32_t qrope = smem_u32(sm + kQRope);
      const uint32_t qtail = smem_u32(sm + kQTail);
      const uint32_t kvbase = smem_u32(sm + kKV);
      bool dead = false;
      for (int rnd = 0, id = item_of(0, cluster_id, p.nclusters); id < total_items && !dead;
           id = item_of(++rnd, cluster_id, p.nclusters)) {
        const Item it = decode_item(plan, ord, obase, a.batch, id);
        if (!mbar_wait<false>(&bars[B_Q_FULL], qi & 1, abort, limit) ||
            !mbar_wait<false>(&bars[B_QT_FULL], qi & 1, abort, limit))
          break;
        ++qi;
        tc_fence_after();
        const uint32_t kb0 = kb;
        // Two independent streams, polled without blocking: S_j = Q K_j^T
        // as soon as key block j has landed and a score buffer is free, and
        // O += P_j V_j as soon as P_j is written (own rows by the softmax,
        // the other rows by the receivers). Waiting for P_j before issuing
        // the next scores would tie every block to the softmax two blocks back.
        int nq = 0, np = 0;
        bool ofree = false;
        uint64_t idle_since = 0;
        while (np < it.nblocks) {
          bool did = false;
          if (nq < it.nblocks) {
            const uint32_t kbi = kb0 + nq;
            const uint32_t s = kbi % kStages, sb = sc & 1, ph = (kbi / kStages) & 1;
            bool landed = mbar_test_wait(&bars[B_S_EMPTY0 + sb], ((sc >> 1) & 1) ^ 1);
#pragma unroll
            for (int w = 0; w < kProducers; ++w)
              landed = landed && mbar_test_wait(&bars[B_KV_FULL0 + s * kProducers + w], ph);
            if (landed) {
              tc_fence_after();
              const uint32_t stg = kvbase + s * kKVStage;
              const uint32_t d = tmem + kTmemS + 64 * sb;
#pragma unroll
              for (int k = 0; k < kQTmemSteps; ++k)  // latent dims 16k.. from TMEM, keys' 64-dim chunk k/4
                mma_bf16_ts(d, tmem + kTmemQ + 8 * k,
                            smem_desc(stg + (k >> 2) * kKVLat + 32 * (k & 3), 16, 1024, kSwizzle128B),
                            idesc_qk, k != 0);
#pragma unroll
              for (int k = kQTmemSteps; k < 16; ++k)  // latent dims 224..255 from shared memory
                mma_bf16_ss(d, smem_desc(qtail + 32 * (k - kQTmemSteps), 16, 512, kSwizzle64B),
                            smem_desc(stg + (k >> 2) * kKVLat + 32 * (k & 3), 16, 1024, kSwizzle128B),
                            idesc_qk, 1);
#pragma unroll
              for (int t = 0; t < 2; ++t)
                mma_bf16_ss(d, smem_desc(qrope + 32 * t, 16, 512, kSwizzle64B),
                            smem_desc(stg + 4 * kKVLat + 32 * t, 16, 512, kSwizzle64B), idesc_qk, 1);
              mma_commit(&bars[B_S_FULL0 + sb]);
              TC_TRACE(true, TR_MMA, kbi, 0);
              ++sc;
              if (++nq == it.nblocks) mma_commit(&bars[B_Q_EMPTY]);  // last use of Q
              did = true;
            }
          }
          if (np < nq) {
            if (!ofree) ofree = mbar_test_wait(&bars[B_O_FREE], (ii & 1) ^ 1);
            const uint32_t pb = pc & 1;
            if (ofree && mbar_test_wait(&bars[B_P_FULL0 + pb], (pc >> 1) & 1)) {
              tc_fence_after();
              const uint32_t s = (kb0 + np) % kStages;
              const uint32_t stg = kvbase + s * kKVStage;
#pragma unroll
              for (int t = 0; t < BN / 16; ++t)
                mma_bf16_ts(tmem + kTmemO, tmem + tmem_p_col(pb, t),
                            smem_desc(stg + t * 2048, kKVLat, 1024, kSwizzle128B), idesc_pv,
                            (np | t) != 0);
              mma_commit(&bars[B_KV_EMPTY0 + s]);
              mma_commit(&bars[B_O_DONE0 + pb]);
              TC_TRACE(true, TR_MMA, kb0 + np, 1);
              ++pc;
              ++np;
              did = true;
            }
          }
          if (did) {
            idle_since = 0;
          } else {  // nothing ready: bounded like every other wait
            if (*abort) {
              dead = true;
              break;
            }
            const uint64_t now = global_timer_ns();
            if (idle_since == 0) idle_since = now;
            else if (now - idle_since > limit) {
              *abort = 1;
              dead = true;
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
  } else if (!own_quarter && wg == 0) {
    // ------------------------------------------------------------ score senders
    // Thread rp owns tile row 64 (1 - c) + rp, which the peer's softmax
    // runs. Per item it writes that row's latent query half into TMEM (QK's
    // A operand); per block it reads the row's fp32 partial score from TMEM,
    // scales it into the log2 domain (-inf for a column the byte-form mask
    // hides) and stores it into the peer's SX buffer, whose arrival
    // completes the peer's SX_FULL.
    const int rp = (q4 - 2 * (int)(1u - cta)) * 32 + lane;
    const int r = 64 * (int)(1u - cta) + rp;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const float scale2 = a.sm_scale * kLog2e;
    const uint32_t sx_peer = mapa(smem_u32(sm + kSX + rp * 16), peer);
    const uint32_t sxfull_peer0 = mapa(smem_u32(&bars[B_SX_FULL0]), peer);
    const bool tr = warp == (int)(2 - 2 * cta) && lane == 0;  // traced thread
    (void)tr;
    uint32_t g = 0, qi = 0;
    bool dead = false;
    cluster_wait();  // the peer's barriers are initialised
    for (int rnd = 0, id = item_of(0, cluster_id, p.nclusters); id < total_items;
         id = item_of(++rnd, cluster_id, p.nclusters)) {
      const Item it = decode_item(plan, ord, obase, a.batch, id);
      {
        // Row r of the query tile, this CTA's 256 latent dims, into TMEM as
        // bf16 pairs once the previous item's last QK is done. Rows past
        // the last query row read as zeros.
        const int64_t qrow = (int64_t)it.q0 * H + it.row0 + r;
        const uint4* src = reinterpret_cast<const uint4*>(a.q + qrow * kDqk + 256 * cta);
        const bool in = qrow < q_rows;
        if (!dead) dead = !mbar_wait<false>(&bars[B_Q_EMPTY], (qi & 1) ^ 1, abort, limit);
        ++qi;
        tc_fence_after();
        {  // dims 0..127, then 128..223
          uint4 v[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) v[k] = in ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
          uint32_t w0[32], w1[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            w0[4 * k] = v[k].x; w0[4 * k + 1] = v[k].y; w0[4 * k + 2] = v[k].z; w0[4 * k + 3] = v[k].w;
            w1[4 * k] = v[8 + k].x; w1[4 * k + 1] = v[8 + k].y;
            w1[4 * k + 2] = v[8 + k].z; w1[4 * k + 3] = v[8 + k].w;
          }
          tmem_st32(tmem + lane_base + kTmemQ, w0);
          tmem_st32(tmem + lane_base + kTmemQ + 32, w1);
        }
        {
          uint4 v[12];
#pragma unroll
          for (int k = 0; k < 12; ++k) v[k] = in ? __ldg(src + 16 + k) : make_uint4(0, 0, 0, 0);
          uint32_t w0[32], w1[16];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            w0[4 * k] = v[k].x; w0[4 * k + 1] = v[k].y; w0[4 * k + 2] = v[k].z; w0[4 * k + 3] = v[k].w;
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            w1[4 * k] = v[8 + k].x; w1[4 * k + 1] = v[8 + k].y;
            w1[4 * k + 2] = v[8 + k].z; w1[4 * k + 3] = v[8 + k].w;
          }
          tmem_st32(tmem + lane_base + kTmemQ + 64, w0);
          tmem_st16(tmem + lane_base + kTmemQ + 96, w1);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();  // one arrival per warp: the warp's TMEM accesses are collective
        if (lane == 0) mbar_arrive(&bars[B_QT_FULL]);
      }
      // Byte-form mask (the bit form is applied by the owner's softmax): the
      // bytes of a block arrive as (draft node, 8-column group) pairs over
      // the nodes of the peer's rows; sender thread rp owns pairs rp + 64 k,
      // held one block ahead when they are few enough. Row r's hidden
      // columns are sent as -inf.
      const int rows_req = it.n * H;
      const int node = (it.row0 + r < rows_req ? it.row0 + r : rows_req - 1) / H;
      const int pre = kSkip ? it.L - it.n : 0;  // prefix columns: visible, mask unread
      const int peer0 = it.row0 + 64 * (int)(1u - cta);
      const int i_lo = min(peer0, rows_req - 1) / H;
      const int cnt = max(1, min(it.n - 1, (peer0 + kOwnRows - 1) / H) - i_lo + 1);
      constexpr int kGroups = BN / 8;  // 8-column groups per block row
      const int pairs = cnt * kGroups;
      const bool prefetch = pairs <= kOwnRows * kMaskPrefetch;
      uint8_t raw[kMaskPrefetch][8];
      auto load_mask = [&](int blk_) {
        const int jb_ = it.j0 + blk_ * BN;
#pragma unroll
        for (int k = 0; k < kMaskPrefetch; ++k) {
          const int q = rp + kOwnRows * k;
          if (q < pairs) {
            const int pos0 = jb_ + 8 * (q % kGroups);
            const uint8_t* src = a.mask + it.mask0 + (int64_t)(i_lo + q / kGroups) * it.L + pos0;
#pragma unroll
            for (int e = 0; e < 8; ++e)
              raw[k][e] = pos0 + e < it.j1 && (!kSkip || pos0 + e >= pre) ? __ldg(src + e) : 0;
          }
        }
      };
      if (!kBits && prefetch) load_mask(0);
      for (int blk = 0; blk < it.nblocks; ++blk, ++g) {
        const uint32_t b = g & 1, ph = (g >> 1) & 1;
        uint64_t vm = ~0ull;
        if constexpr (!kBits) {
          const int jb = it.j0 + blk * BN;
          uint8_t* vb = reinterpret_cast<uint8_t*>(vis + b * kVisNodes);
          if (prefetch) {
#pragma unroll
            for (int k = 0; k < kMaskPrefetch; ++k) {
              const int q = rp + kOwnRows * k;
              if (q < pairs) {
                uint32_t bits = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) bits |= (raw[k][e] != 0 ? 1u : 0u) << e;
                vb[(q / kGroups) * 8 + q % kGroups] = (uint8_t)bits;
              }
            }
            if (blk + 1 < it.nblocks) load_mask(blk + 1);
          } else {
            for (int q = rp; q < pairs; q += kOwnRows) {
              const int pos0 = jb + 8 * (q % kGroups);
              const uint8_t* src = a.mask + it.mask0 + (int64_t)(i_lo + q / kGroups) * it.L + pos0;
              uint32_t bits = 0;
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (pos0 + e < it.j1 && (!kSkip || pos0 + e >= pre) && __ldg(src + e)) bits |= 1u << e;
              vb[(q / kGroups) * 8 + q % kGroups] = (uint8_t)bits;
            }
          }
          named_bar_sync(3, kOwnRows);  // the two sender warps
          const int ni = node - i_lo;
          vm = (ni >= 0 && ni < cnt) ? vis[b * kVisNodes + ni] : 0ull;
          if (kSkip && pre > jb) {  // the block's prefix columns, up to the split's end
            const int pc = min(pre, it.j1) - jb;
            vm |= pc >= 64 ? ~0ull : (1ull << pc) - 1ull;
          }
        }
        if (!dead) dead = !mbar_wait<false>(&bars[B_S_FULL0 + b], ph, abort, limit);
        TC_TRACE(tr, TR_SENDER, g, 0);
        tc_fence_after();
        uint32_t s0[32], s1[16];
        const uint32_t tsrc = tmem + lane_base + kTmemS + 64 * b;
        tmem_ld32_nw(tsrc, s0);
        tmem_ld16_nw(tsrc + 32, s1);
        tmem_ld_wait();
        tmem_regs_ready(s0);
        tmem_regs_ready(s1);
        tc_fence_before();
        __syncwarp();  // one arrival per warp: the warp's TMEM accesses are collective
        if (lane == 0) mbar_arrive(&bars[B_S_EMPTY0 + b]);  // the score buffer may take block g+2
        float x[BN];
#pragma unroll
        for (int c = 0; c < BN; ++c)
          x[c] = (vm >> c) & 1ull ? __uint_as_float(c < 32 ? s0[c] : s1[c - 32]) * scale2 : -INFINITY;
        // the peer's softmax has read block g-2 from this buffer
        if (!dead) dead = !mbar_wait<false>(&bars[B_SX_FREE0 + b], ph ^ 1, abort, limit);
        if (!dead && !*abort) {
          const uint32_t dst = sx_peer + b * kSXBytes;
          const uint32_t bar = sxfull_peer0 + 8 * b;
#pragma unroll
          for (int q = 0; q < BN / 4; ++q)
            st_async_v4(dst + kXChunk * q, __float_as_uint(x[4 * q]), __float_as_uint(x[4 * q + 1]),
                        __float_as_uint(x[4 * q + 2]), __float_as_uint(x[4 * q + 3]), bar);
        }
        TC_TRACE(tr, TR_SENDER, g, 1);
      }
    }
  } else if (!own_quarter) {  // wg == 1
    // ------------------------------------------------------------ P receivers
    // Thread rp owns tile row 64 (1 - c) + rp. Per block it takes that row's
    // P (bf16), running max and quarter sums from the peer's message, rescales
    // this CTA's half of the row of O when the max moved, and writes P into
    // TMEM for the P.V MMA. After an item it writes the row's output half.
    const int rp = (q4 - 2 * (int)(1u - cta)) * 32 + lane;
    const int r = 64 * (int)(1u - cta) + rp;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const uint32_t t_o = tmem + lane_base + kTmemO;
    const uint32_t pxfree_peer0 = mapa(smem_u32(&bars[B_PX_FREE0]), peer);
    const bool arms = warp == (int)(6 - 2 * cta) && lane == 0;  // re-arms PX_FULL
    uint32_t g = 0;
    bool dead = false;
    // the P.V of block x has completed (it read P buffer x & 1)
    auto wait_pv = [&](uint32_t x) {
      if (!dead) dead = !mbar_wait<false>(&bars[B_O_DONE0 + (x & 1)], (x >> 1) & 1, abort, limit);
    };
    cluster_wait();
    for (int rnd = 0, id = item_of(0, cluster_id, p.nclusters); id < total_items;
         id = item_of(++rnd, cluster_id, p.nclusters)) {
      const Item it = decode_item(plan, ord, obase, a.batch, id);
      float m_prev = -INFINITY, lsum = 0.f;
      for (int blk = 0; blk < it.nblocks; ++blk, ++g) {
        const uint32_t b = g & 1, ph = (g >> 1) & 1;
        if (!dead) dead = !mbar_wait<true>(&bars[B_PX_FULL0 + b], ph, abort, limit);
        TC_TRACE(arms, TR_RECEIVER, g, 0);
        const uint8_t* px = sm + kPX + b * kPXBytes + rp * 8;
        uint32_t pk[BN / 2];
#pragma unroll
        for (int q = 0; q < BN / 4; ++q) {
          const uint2 u = *reinterpret_cast<const uint2*>(px + kPChunk * q);
          pk[2 * q] = u.x;
          pk[2 * q + 1] = u.y;
        }
        uint2 ml[kRowThreads];  // (m, l_h) from each of the owner's four threads
#pragma unroll
        for (int q = 0; q < kRowThreads; ++q) ml[q] = *reinterpret_cast<const uint2*>(px + kPChunk * (BN / 4 + q));
        __syncwarp();
        if (lane == 0 && !dead && !*abort) {
          if (arms) mbar_arrive_expect_tx(&bars[B_PX_FULL0 + b], kPXTx);  // block g+2
          mbar_arrive_remote_relaxed(pxfree_peer0 + 8 * b);
        }
        const float m_new = __uint_as_float(ml[0].x);
        lsum = (__uint_as_float(ml[0].y) + __uint_as_float(ml[1].y)) +
               (__uint_as_float(ml[2].y) + __uint_as_float(ml[3].y));
        // the owner rescales its half of O by exactly this factor: same
        // inputs to the same instruction
        const bool resc = blk > 0 && __float_as_uint(m_new) != __float_as_uint(m_prev);
        const float corr = resc ? ex2_approx(m_prev - m_new) : 1.f;
        m_prev = m_new;
        // P buffer g & 1 was last read by the P.V of block g - 2; a rescale
        // of O also needs the P.V of block g - 1 to be done
        const bool any_resc = __any_sync(0xffffffffu, resc);
        if (any_resc) wait_pv(g - 1);
        else if (blk >= 2) wait_pv(g - 2);
        TC_TRACE(arms, TR_RECEIVER, g, 1);
        tc_fence_after();
        if (any_resc) {
#pragma unroll 1
          for (int k = 0; k < 8; ++k) {
            uint32_t o[32];
            tmem_ld32(t_o + 32 * k, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            tmem_st32(t_o + 32 * k, o);
          }
        }
        {
          uint32_t p01[16], p2[8];
#pragma unroll
          for (int c = 0; c < 16; ++c) p01[c] = pk[c];
#pragma unroll
          for (int c = 0; c < 8; ++c) p2[c] = pk[16 + c];
          tmem_st16(tmem + lane_base + tmem_p_col(g & 1, 0), p01);
          tmem_st8(tmem + lane_base + tmem_p_col(g & 1, 2), p2);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();  // one arrival per warp: the warp's TMEM accesses are collective
        if (lane == 0) mbar_arrive(&bars[B_P_FULL0 + (g & 1)]);
        TC_TRACE(arms, TR_RECEIVER, g, 2);
      }
      // epilogue: this CTA's 256 value dims of the row, divided by the
      // owner's final sum, once the item's last P.V is done
      wait_pv(g - 1);
      tc_fence_after();
      const float l = lsum;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int rows_req = it.n * H;
      const bool valid = it.row0 + r < rows_req;
      const int64_t grow = (int64_t)it.q0 * H + it.row0 + r;
#pragma unroll 1
      for (int k = 0; k < 8; ++k) {
        uint32_t o[32];
        tmem_ld32(t_o + 32 * k, o);
        if (!valid) continue;
        if (it.splits == 1) {
          uint4* dst = reinterpret_cast<uint4*>(a.out + grow * kDv + 256 * cta + 32 * k);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(o[8 * v + 2 * e]) * inv,
                                                              __uint_as_float(o[8 * v + 2 * e + 1]) * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(a.ws_o + ((int64_t)it.split * R + grow) * kDv +
                                                  256 * cta + 32 * k);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                 __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
        }
      }
      tc_fence_before();
      __syncwarp();  // one arrival per warp: the warp's TMEM accesses are collective
      if (lane == 0) mbar_arrive(&bars[B_O_FREE]);  // O has been read: the next item may overwrite it
      TC_MARK(arms, 7);
    }
  } else {
    // ------------------------------------------------------------ softmax, epilogue (own rows)
    // Four threads per own row, in the four warps of the row's lane quarter:
    // thread h takes columns [12 h, 12 h + 12) of every block and dims
    // [64 h, 64 h + 64) of this CTA's half of O. Block g's peer partials
    // arrive in SX buffer g & 1; the row's P goes to this CTA's TMEM and to
    // the peer's PX buffer g & 1.
    const int h = wg;
    const int ro = (q4 - 2 * (int)cta) * 32 + lane;
    const int r = 64 * (int)cta + ro;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const uint32_t t_o = tmem + lane_base + kTmemO + 64 * h;
    const uint32_t sxfree_peer0 = mapa(smem_u32(&bars[B_SX_FREE0]), peer);
    const uint32_t px_peer = mapa(smem_u32(sm + kPX + ro * 8), peer);
    const uint32_t pxfull_peer0 = mapa(smem_u32(&bars[B_PX_FULL0]), peer);
    const bool arms = warp == (int)(2 * cta) && lane == 0;   // re-arms SX_FULL
    const int quad_bar = 1 + (q4 & 1);                       // the rows' four warps (128 threads)
    const float scale2 = a.sm_scale * kLog2e;
    uint32_t g = 0, qi = 0;
    bool dead = false;
    cluster_wait();  // the peer's barriers are initialised
    // the P.V of block x has completed (it read P buffer x & 1)
    auto wait_pv = [&](uint32_t x) {
      if (!dead) dead = !mbar_wait<false>(&bars[B_O_DONE0 + (x & 1)], (x >> 1) & 1, abort, limit);
    };

    // this row's share of the query's latent dims 0..223 into TMEM for item
    // `id`: thread h writes dims [56 h, 56 h + 56), TMEM columns
    // [28 h, 28 h + 28) of the query block
    auto load_q = [&](int id) {
      const Item it = decode_item(plan, ord, obase, a.batch, id);
      const int64_t qrow = (int64_t)it.q0 * H + it.row0 + r;
      const uint4* src = reinterpret_cast<const uint4*>(a.q + qrow * kDqk + 256 * cta + 56 * h);
      const bool in = qrow < q_rows;
      uint4 v[7];
#pragma unroll
      for (int k = 0; k < 7; ++k) v[k] = in ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
      if (!dead) dead = !mbar_wait<false>(&bars[B_Q_EMPTY], (qi & 1) ^ 1, abort, limit);
      ++qi;
      tc_fence_after();
      uint32_t w[28];
#pragma unroll
      for (int k = 0; k < 7; ++k) {
        w[4 * k] = v[k].x; w[4 * k + 1] = v[k].y; w[4 * k + 2] = v[k].z; w[4 * k + 3] = v[k].w;
      }
      const uint32_t tq = tmem + lane_base + kTmemQ + 28 * h;
      switch (h) {  // pieces of 16, 8 and 4 columns, each at a multiple of its width
        case 0: tmem_st_q28<0, 16, 24>(tq, w); break;
        case 1: tmem_st_q28<4, 20, 0>(tq, w); break;
        case 2: tmem_st_q28<8, 0, 24>(tq, w); break;
        default: tmem_st_q28<12, 4, 0>(tq, w); break;
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();  // one arrival per warp: the warp's TMEM accesses are collective
      if (lane == 0) mbar_arrive(&bars[B_QT_FULL]);
    };

    int id = item_of(0, cluster_id, p.nclusters);
    if (id < total_items) load_q(id);
    for (int rnd = 0; id < total_items; id = item_of(++rnd, cluster_id, p.nclusters)) {
      const Item it = decode_item(plan, ord, obase, a.batch, id);
      const int rows_req = it.n * H;
      const int row = it.row0 + r;
      const bool valid = row < rows_req;
      const int node = (valid ? row : rows_req - 1) / H;
      const int pre = kSkip ? it.L - it.n : 0;  // prefix columns: visible, mask unread
      // Bit-form mask: this row's node reads the (up to) three words holding
      // a block's 48 columns straight from global memory, one block ahead.
      // (With the byte form the score senders apply the mask: hidden columns
      // arrive as -inf in the peer's partial scores.)
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
      float m = -INFINITY, lh = 0.f;
      for (int blk = 0; blk < it.nblocks; ++blk, ++g) {
        const uint32_t b = g & 1, ph = (g >> 1) & 1;
        const int jb = it.j0 + blk * BN;
        TC_TRACE(arms, TR_SOFTMAX, g, 8);
        uint32_t vh = 0;  // visibility of the thread's 12 columns (bit form)
        if constexpr (kBits) {
          const uint32_t w0 = mnext[0], w1 = mnext[1], w2 = mnext[2];
          if (blk + 1 < it.nblocks) load_bits(blk + 1);
          const int o = jb & 31;
          const uint64_t lo = (uint64_t)w0 | ((uint64_t)w1 << 32);
          uint64_t vm = o ? (lo >> o) | ((uint64_t)w2 << (64 - o)) : lo;
          const int lim = it.j1 - jb;  // columns of this block inside the split
          if (lim < 64) vm &= (1ull << lim) - 1ull;
          if (kSkip && pre > jb) {  // the block's prefix columns, up to the split's end
            const int pc = min(pre, it.j1) - jb;
            vm |= pc >= 64 ? ~0ull : (1ull << pc) - 1ull;
          }
          vh = (uint32_t)(vm >> (kQCols * h)) & ((1u << kQCols) - 1u);
        }
        TC_TRACE(arms, TR_SOFTMAX, g, 9);

        // this CTA's partial scores of the row's 12 columns, from TMEM
        if (!dead) dead = !mbar_wait<false>(&bars[B_S_FULL0 + b], ph, abort, limit);
        TC_TRACE(arms, TR_SOFTMAX, g, 0);
        tc_fence_after();
        // naturally aligned pieces from column 12 h, one wait: 8 + 4 columns
        // for even h, 4 + 8 for odd h
        uint32_t own[kQCols];
        {
          const uint32_t tsrc = tmem + lane_base + kTmemS + 64 * b + kQCols * h;
          uint32_t x8[8], x4[4];
          if ((h & 1) == 0) {
            tmem_ld8_nw(tsrc, x8);
            tmem_ld4_nw(tsrc + 8, x4);
          } else {
            tmem_ld4_nw(tsrc, x4);
            tmem_ld8_nw(tsrc + 4, x8);
          }
          tmem_ld_wait();
          tmem_regs_ready(x8);
          tmem_regs_ready(x4);
          if ((h & 1) == 0) {
#pragma unroll
            for (int c = 0; c < 8; ++c) own[c] = x8[c];
#pragma unroll
            for (int c = 0; c < 4; ++c) own[8 + c] = x4[c];
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) own[c] = x4[c];
#pragma unroll
            for (int c = 0; c < 8; ++c) own[4 + c] = x8[c];
          }
        }
        tc_fence_before();
        __syncwarp();  // one arrival per warp: the warp's TMEM accesses are collective
        if (lane == 0) mbar_arrive(&bars[B_S_EMPTY0 + b]);
        // the peer's partials of the same columns (already in the log2 domain)
        if (!dead) dead = !mbar_wait<true>(&bars[B_SX_FULL0 + b], ph, abort, limit);
        TC_TRACE(arms, TR_SOFTMAX, g, 1);
        const uint8_t* sx = sm + kSX + b * kSXBytes + ro * 16 + kXChunk * (kQCols / 4) * h;
        float s[kQCols];
#pragma unroll
        for (int q = 0; q < kQCols / 4; ++q) {
          const float4 v = *reinterpret_cast<const float4*>(sx + kXChunk * q);
          const float pv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 4 * q + e;
            s[c] = fmaf(__uint_as_float(own[c]), scale2, pv[e]);
          }
        }
        __syncwarp();
        if (lane == 0 && !dead && !*abort) {
          if (arms) mbar_arrive_expect_tx(&bars[B_SX_FULL0 + b], kSXTx);  // block g+2
          mbar_arrive_remote_relaxed(sxfree_peer0 + 8 * b);
        }

        // masked maximum of the quarter row, then of the row
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < kQCols; ++c) {
          if constexpr (kBits) s[c] = (vh >> c) & 1u ? s[c] : -INFINITY;
          mx4[c & 3] = fmaxf(mx4[c & 3], s[c]);
        }
        const float mxh = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        float* mrow = mxs + (b * kOwnRows + ro) * kRowThreads;
        mrow[h] = mxh;
        named_bar_sync(quad_bar, 128);
        TC_TRACE(arms, TR_SOFTMAX, g, 2);
        const float4 m4 = *reinterpret_cast<const float4*>(mrow);
        const float mb = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));
        float corr = 1.f;
        bool resc = false;
        if (mb > m + kRescale) {
          corr = ex2_approx(m - mb);
          m = mb;
          resc = true;
        }
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[kQCols / 2];
        if (m == -INFINITY) {
#pragma unroll
          for (int c = 0; c < kQCols / 2; ++c) pk[c] = 0u;
        } else {
#pragma unroll
          for (int c = 0; c < kQCols / 2; ++c) {
            const float p0 = ex2_approx(s[2 * c] - m), p1 = ex2_approx(s[2 * c + 1] - m);
            const __nv_bfloat162 v = __floats2bfloat162_rn(p0, p1);
            // the denominator sums the same bf16 weights the P.V product uses,
            // so O / l stays a true weighted average of the value rows
            rs4[c & 3] += __low2float(v) + __high2float(v);
            pk[c] = *reinterpret_cast<const uint32_t*>(&v);
          }
        }
        lh = lh * corr + ((rs4[0] + rs4[1]) + (rs4[2] + rs4[3]));
        TC_TRACE(arms, TR_SOFTMAX, g, 6);

        // the row's quarter of P, the running max and this quarter's sum to
        // the peer, once its receivers have taken block g-2 from that buffer
        if (!dead) dead = !mbar_wait<true>(&bars[B_PX_FREE0 + b], ph ^ 1, abort, limit);
        TC_TRACE(arms, TR_SOFTMAX, g, 7);
        if (!dead && !*abort) {
          const uint32_t dst = px_peer + b * kPXBytes;
          const uint32_t bar = pxfull_peer0 + 8 * b;
#pragma unroll
          for (int q = 0; q < kQCols / 4; ++q)
            st_async_v2(dst + kPChunk * (3 * h + q), pk[2 * q], pk[2 * q + 1], bar);
          st_async_v2(dst + kPChunk * (BN / 4 + h), __float_as_uint(m), __float_as_uint(lh), bar);
        }
        TC_TRACE(arms, TR_SOFTMAX, g, 3);

        // P buffer g & 1 was last read by the P.V of block g - 2; a rescale
        // of O also needs the P.V of block g - 1 to be done
        const bool need = resc && blk > 0;
        const bool any_need = __any_sync(0xffffffffu, need);
        if (any_need) wait_pv(g - 1);
        else if (blk >= 2) wait_pv(g - 2);
        TC_TRACE(arms, TR_SOFTMAX, g, 4);
        tc_fence_after();
        if (any_need) {
          const float f = need ? corr : 1.f;
#pragma unroll 1
          for (int k = 0; k < 2; ++k) {
            uint32_t o[32];
            tmem_ld32(t_o + 32 * k, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32(t_o + 32 * k, o);
          }
        }
        // the quarter's 6 bf16 pairs (keys 12h .. 12h+11) at P word 6h of the
        // buffer: pieces of 4 and 2 columns, each at a multiple of its width
        {
          const uint32_t pb = g & 1;
          uint32_t x4[4], x2[2];
          if ((h & 1) == 0) {
#pragma unroll
            for (int c = 0; c < 4; ++c) x4[c] = pk[c];
            x2[0] = pk[4];
            x2[1] = pk[5];
            const uint32_t c4 = h == 0 ? tmem_p_col(pb, 0) : tmem_p_col(pb, 1) + 4;
            const uint32_t c2 = h == 0 ? tmem_p_col(pb, 0) + 4 : tmem_p_col(pb, 2);
            tmem_st4(tmem + lane_base + c4, x4);
            tmem_st2(tmem + lane_base + c2, x2);
          } else {
            x2[0] = pk[0];
            x2[1] = pk[1];
#pragma unroll
            for (int c = 0; c < 4; ++c) x4[c] = pk[2 + c];
            const uint32_t c2 = h == 1 ? tmem_p_col(pb, 0) + 6 : tmem_p_col(pb, 2) + 2;
            const uint32_t c4 = h == 1 ? tmem_p_col(pb, 1) : tmem_p_col(pb, 2) + 4;
            tmem_st2(tmem + lane_base + c2, x2);
            tmem_st4(tmem + lane_base + c4, x4);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();  // one arrival per warp: the warp's TMEM accesses are collective
        if (lane == 0) mbar_arrive(&bars[B_P_FULL0 + (g & 1)]);
        TC_TRACE(arms, TR_SOFTMAX, g, 5);
      }

      // the next item's query (QK may start on it while this epilogue runs)
      const int next = item_of(rnd + 1, cluster_id, p.nclusters);
      if (next < total_items) load_q(next);

      // epilogue: O / l for the row's 64 dims of this CTA's half, and the LSE
      lxs[ro * kRowThreads + h] = lh;
      named_bar_sync(quad_bar, 128);
      const float4 l4 = *reinterpret_cast<const float4*>(lxs + ro * kRowThreads);
      const float l = (l4.x + l4.y) + (l4.z + l4.w);
      wait_pv(g - 1);  // the item's last P.V
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t grow = (int64_t)it.q0 * H + row;
#pragma unroll 1
      for (int k = 0; k < 2; ++k) {
        uint32_t o[32];
        tmem_ld32(t_o + 32 * k, o);
        if (!valid) continue;
        const int col = 256 * (int)cta + 64 * h + 32 * k;
        if (it.splits == 1) {
          uint4* dst = reinterpret_cast<uint4*>(a.out + grow * kDv + col);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(o[8 * v + 2 * e]) * inv,
                                                              __uint_as_float(o[8 * v + 2 * e + 1]) * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(a.ws_o + ((int64_t)it.split * R + grow) * kDv + col);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                 __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
        }
      }
      if (valid && h == 0) {
        const float lv = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        if (it.splits == 1) a.lse[grow] = lv;
        else a.ws_lse[(int64_t)it.split * R + grow] = lv;
      }
      tc_fence_before();
      __syncwarp();  // one arrival per warp: the warp's TMEM accesses are collective
      if (lane == 0) mbar_arrive(&bars[B_O_FREE]);  // O has been read: the next item may overwrite it
      TC_MARK(arms, 6);
    }
  }

  TC_MARK(tid == 0, 8);
  if (is_producer || is_mma) cluster_wait();  // pairs with the arrival after set-up
  // this CTA's outputs are issued: the merge kernel (launched as a dependent
  // grid) may start its set-up; it waits for this grid's completion before
  // reading any partial
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0 && *abort) {
    flag(a.status, MT_DEV_TIMEOUT);
    // remote stores issued before the give-up land within microseconds
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < kAbortSettleNs) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == mma_warp) {
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
int g_test_drop_item = -1;
unsigned long long g_test_limit_ns = 0;

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

// The instantiations: byte or bit mask, each with and without the prefix skip.
constexpr int kVariants = 4;
KernelFn kernel_variant(int i) {
  switch (i) {
    case 0: return verify_tc_kernel<false, false>;
    case 1: return verify_tc_kernel<false, true>;
    case 2: return verify_tc_kernel<true, false>;
    default: return verify_tc_kernel<true, true>;
  }
}
int variant_index(bool bits, bool skip) { return (bits ? 2 : 0) + (skip ? 1 : 0); }

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

void set_tc_test_hooks(int drop_item, unsigned long long limit_ns) {
  tc::g_test_drop_item = drop_item;
  tc::g_test_limit_ns = limit_ns;
}

cudaError_t launch_verify_tc(const VerifyArgs& a, int num_sms, cudaStream_t stream) {
  using namespace tc;
  if (a.num_slots <= 0 || a.num_slots >= 0x7fffffffLL ||
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
  VerifyArgs full = a;
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
  const KernelFn fn = kernel_variant(variant_index(a.bits_mask != 0, a.skip_prefix != 0));
  // The plan of a launch lives in shared memory: requests go in chunks of
  // kMaxBatch, one launch each, with the indptrs offset to the chunk.
  for (int b0 = 0; b0 < a.batch; b0 += kMaxBatch) {
    TcParams p;
    p.a = full;
    p.a.batch = min(kMaxBatch, a.batch - b0);
    p.a.kv_indptr = a.kv_indptr + b0;
    p.a.qo_indptr = a.qo_indptr + b0;
    p.a.mask_indptr = a.mask_indptr + b0;
    p.nclusters = nclusters;
    p.first_chunk = b0 == 0;
    p.last_chunk = b0 + kMaxBatch >= a.batch;
    p.drop_item = g_test_drop_item;
    p.limit_ns = g_test_limit_ns > 0 ? g_test_limit_ns : sm100::kWaitLimitNs;
    cudaError_t e = cudaLaunchKernelEx(&cfg, fn, p, tq_rope, tkv_lat, tkv_rope);
    if (e != cudaSuccess) return e;
  }
  if (a.max_splits > 1) return launch_lse_merge(full, stream);
  return cudaSuccess;
}

#ifdef MT_TC_TRACE
// Copies the pipeline trace of the last traced launch to host memory.
extern "C" int mla_tree_tc_trace_read(void* host, size_t bytes) {
  if (bytes < sizeof(tc::g_tc_trace)) return -1;
  return cudaMemcpyFromSymbol(host, tc::g_tc_trace, sizeof(tc::g_tc_trace)) == cudaSuccess ? 0 : -1;
}
#endif

int verify_tc_launches(int batch, int total_q, int heads, int max_splits) {
  (void)total_q;
  (void)heads;
  if (batch <= 0) return 0;
  return (batch + tc::kMaxBatch - 1) / tc::kMaxBatch + (max_splits > 1 ? 1 : 0);
}

}  // namespace mt
