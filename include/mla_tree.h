/*
 * mla_tree.h -- C ABI of the GB300 (sm_103a) tree-verify MLA attention library.
 *
 * The operation is the verify step of tree speculative decoding with
 * Multi-head Latent Attention, as described on the pages
 *   "The Moment of Truth: Flipping the Switch on a Custom CUDA Verify Kernel"
 *     (section "The Long Road to Parity": prefix + draft KV marshaling,
 *      mask row stride prefix + draft, the logged shapes q (9, 8, 576),
 *      kv_buf (slots, 576), mask (270,); section "The Broader Context":
 *      KV-split flash-decode, split count, 128-bit KV loads) and
 *   "The Pivot to Live Cutover: A Decision Point in Custom CUDA Kernel
 *     Integration" (section "The Technical Investigation: Probing the
 *      Integration Surface": flat custom mask indexed per sequence by
 *      mask_indptr; latent KV buffer of shape [num_slots, 1, 576] with page
 *      size 1; section "Input Knowledge Required": 512 absorbed-latent + 64
 *      rope query dims, paged KV through kv_indices).
 *
 * Conventions for every entry point
 *   - All array pointers are DEVICE pointers owned by the caller. The library
 *     never allocates, frees, copies to the host or synchronises, so every
 *     call can be recorded into a CUDA graph; only host-known scalars are
 *     validated on the host.
 *   - Work is enqueued on `stream`; the return value reports host-side
 *     argument errors (nothing is launched then) or a launch error.
 *   - Values the host cannot see (indices, parents, indptr contents) are
 *     checked by the kernels: a bad value ORs a MT_DEV_* bit into
 *     *dev_status (when dev_status is not NULL) and the affected work is
 *     skipped -- no trap, no out-of-bounds access.
 *   - bf16 data is passed as raw 16-bit patterns (mt_bf16).
 *   - Layouts are row-major and contiguous unless a stride is given.
 *
 * Notation: batch B requests; request b owns query tokens
 * qo_indptr[b] .. qo_indptr[b+1]-1 (n_b draft nodes), P_b prefix slots and
 * L_b = P_b + n_b key positions; H heads; a pool row is 576 bf16 (512 latent
 * dims then 64 rope dims); the key is the whole row, the value its first 512.
 */
#ifndef MLA_TREE_H
#define MLA_TREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mt_stream_t;  /* == cudaStream_t */
typedef uint16_t mt_bf16;                  /* raw bf16 bits */

/* Host-side status codes (return values). */
enum {
  MT_OK = 0,
  MT_EINVAL = -1,        /* bad pointer, size, alignment or scalar */
  MT_EUNSUPPORTED = -2,  /* valid request the library cannot serve */
  MT_EWORKSPACE = -3,    /* workspace missing, misaligned or too small */
  MT_ECUDA = -4,         /* a CUDA runtime call or launch failed */
  MT_ESCRATCH = -5       /* needs more scratch than mla_tree_verify_noalloc's
                            built-in MT_NOALLOC_SCRATCH_BYTES */
};

/* Device-side status bits, OR-ed into *dev_status by the kernels. */
#define MT_DEV_BAD_SLOT     0x01  /* slot index outside [0, num_slots) */
#define MT_DEV_BAD_PARENT   0x02  /* parent outside [-1, i-1] */
#define MT_DEV_BAD_INDPTR   0x04  /* decreasing indptr, sizes beyond a capacity, or
                                     qo_indptr[batch] != total_q */
#define MT_DEV_TREE_TOO_BIG 0x08  /* a request with more than MT_MAX_TREE draft nodes */
#define MT_DEV_TIMEOUT      0x10  /* a bounded wait inside a kernel gave up */
#define MT_DEV_MISMATCH     0x20  /* validate mode: the two kernels disagree beyond the tolerance */

#define MT_D_QK 576
#define MT_D_V 512
#define MT_MAX_TREE 8192          /* draft nodes per request for tree_mask_pack */
#define MT_MAX_SPLITS 1024

/* Version of this ABI (major * 100 + minor). */
int mla_tree_abi_version(void);

/* Short English text for a host status code. */
const char* mla_tree_status_string(int status);

/*
 * Draft-KV scatter ("Flipping the Switch", "The Long Road to Parity": the
 * draft tokens' KV arrives as separate tensors and is written to
 * out_cache_loc). For t < total_q:
 *     kv_buf[out_cache_loc[t], 0:576] = src[t * src_row_stride + 0 : +576]
 * bit for bit. src: bf16 [total_q, >=576] with row stride src_row_stride
 * elements (>= 576); kv_buf: bf16 [num_slots, 576]. out_cache_loc entries
 * must be distinct (duplicates leave the written row unspecified). A slot
 * outside [0, num_slots) sets MT_DEV_BAD_SLOT and that row is skipped.
 * 16-byte aligned src/kv_buf with src_row_stride % 8 == 0 take 128-bit
 * copies; other layouts take a 16-bit copy path.
 */
int mla_tree_draft_kv_scatter(const mt_bf16* src, int64_t src_row_stride,
                              const int32_t* out_cache_loc, int total_q,
                              mt_bf16* kv_buf, int64_t num_slots,
                              int32_t* dev_status, mt_stream_t stream);

/*
 * KV index marshaling ("Flipping the Switch", "The Long Road to Parity":
 * the full index array is the prefix slots followed by the draft tokens'
 * slot locations). Writes
 *     kv_indptr[b] = prefix_indptr[b] + qo_indptr[b]          (b = 0..batch)
 *     kv_indices[kv_indptr[b] + j] = prefix_indices[prefix_indptr[b] + j]   j < P_b
 *     kv_indices[kv_indptr[b] + P_b + k] = out_cache_loc[qo_indptr[b] + k] k < n_b
 * prefix_indices: int32 [prefix_indices_len]; prefix_indptr, qo_indptr:
 * int32 [batch+1], non-decreasing, starting at 0; kv_indices: int32
 * [kv_indices_capacity]; kv_indptr: int32 [batch+1].
 * A request that would read past prefix_indices_len or write past the
 * capacity, or decreasing indptrs, sets MT_DEV_BAD_INDPTR and that request's
 * indices are not written.
 */
int mla_tree_kv_indices_build(const int32_t* prefix_indices, int64_t prefix_indices_len,
                              const int32_t* prefix_indptr,
                              const int32_t* out_cache_loc, const int32_t* qo_indptr,
                              int batch, int total_q,
                              int32_t* kv_indices, int64_t kv_indices_capacity,
                              int32_t* kv_indptr,
                              int32_t* dev_status, mt_stream_t stream);

/*
 * Tree mask packing ("Flipping the Switch", "The Long Road to Parity": mask
 * row stride = prefix + draft, the logged mask (270,) = 9 x 30; "Pivot to
 * Live Cutover", "The Technical Investigation": one flat buffer offset per
 * sequence by mask_indptr).
 *   parents: int32 [total_q]; parents[qo_indptr[b] + i] is the local index of
 *            node i's parent in request b, or -1 when node i hangs off the
 *            prefix; nodes are in topological order (parent < i).
 *   kv_indptr: int32 [batch+1] as written by mla_tree_kv_indices_build.
 * Writes mask_indptr: int64 [batch+1], mask_indptr[b+1] = mask_indptr[b] +
 * n_b * L_b, and packed_mask: uint8 [mask_indptr[batch]], row i of request b
 * at mask_indptr[b] + i * L_b holding L_b bytes: 1 for every prefix column
 * and for draft column P_b + k when k is i or an ancestor of i, else 0.
 * A parent out of range sets MT_DEV_BAD_PARENT (the walk stops there); a
 * request with more than MT_MAX_TREE nodes sets MT_DEV_TREE_TOO_BIG; a
 * mask larger than mask_capacity bytes or inconsistent indptrs set
 * MT_DEV_BAD_INDPTR; the affected rows are not written.
 */
int tree_mask_pack(const int32_t* parents, const int32_t* qo_indptr, const int32_t* kv_indptr,
                   int batch, int total_q,
                   int64_t* mask_indptr, uint8_t* packed_mask, int64_t mask_capacity,
                   int32_t* dev_status, mt_stream_t stream);

/*
 * The same tree mask, one bit per (row, column) ("Pivot to Live Cutover",
 * "The Technical Investigation": the custom mask is called a packed
 * bitmask). Row i of request b holds its L_b visibility bits in
 * W_b = ceil(L_b / 32) uint32 words, column j in bit j % 32 of word j / 32
 * (least significant bit first); bits past L_b are 0. Writes
 * mask_word_indptr: int64 [batch+1], mask_word_indptr[b+1] =
 * mask_word_indptr[b] + n_b * W_b, and mask_words: uint32
 * [mask_word_indptr[batch]], row i of request b at mask_word_indptr[b] +
 * i * W_b. Visibility, arguments and error behaviour are those of
 * tree_mask_pack, with mask_capacity_words counted in words. The bit form
 * is an eighth of the bytes and lets the verify kernels read a block's
 * visibility with a few word loads per row.
 */
int tree_mask_pack_bits(const int32_t* parents, const int32_t* qo_indptr, const int32_t* kv_indptr,
                        int batch, int total_q,
                        int64_t* mask_word_indptr, uint32_t* mask_words,
                        int64_t mask_capacity_words,
                        int32_t* dev_status, mt_stream_t stream);

/*
 * The three marshaling steps of one verify step in one launch: exactly the
 * effect of mla_tree_draft_kv_scatter(draft_kv, ...), then
 * mla_tree_kv_indices_build(...) and tree_mask_pack_bits(...) with the
 * kv_indptr it writes, on the same arguments (see those entry points for
 * layouts, capacities and the status bits they set). The three parts run
 * side by side; the mask part takes each request's key count from
 * prefix_indptr and qo_indptr instead of reading kv_indptr. draft_kv and
 * kv_buf must be 16-byte aligned and draft_row_stride a multiple of 8
 * elements, else MT_EINVAL (the separate entry points take any alignment).
 * In "Deploying a Custom sm_120 Verify Kernel into Production" (section
 * "The Context: Why This Deployment Matters") a separate Python backend
 * module wires the kernel into the serving engine and prepares its inputs;
 * here they are one kernel ahead of mla_tree_verify_bits.
 */
int mla_tree_prepare(const mt_bf16* draft_kv, int64_t draft_row_stride,
                     const int32_t* out_cache_loc, const int32_t* prefix_indices,
                     int64_t prefix_indices_len, const int32_t* prefix_indptr,
                     const int32_t* qo_indptr, const int32_t* parents, int batch, int total_q,
                     mt_bf16* kv_buf, int64_t num_slots,
                     int32_t* kv_indices, int64_t kv_indices_capacity, int32_t* kv_indptr,
                     int64_t* mask_word_indptr, uint32_t* mask_words, int64_t mask_capacity_words,
                     int32_t* dev_status, mt_stream_t stream);

/*
 * Bytes of scratch workspace mla_tree_verify needs for these capacities
 * (max_splits 0 = the automatic choice mla_tree_verify makes for 0).
 * Holds the per-token split counts and, when max_splits > 1, the per-split
 * partial outputs (fp32 [splits][total_q*heads][512]) and their LSEs; the
 * caller allocates it once, 256-byte aligned, and may reuse it across calls
 * on one stream.
 */
size_t mla_tree_verify_workspace_bytes(int batch, int total_q, int heads, int max_splits);

/*
 * Number of kernels one mla_tree_verify call with these host scalars
 * launches (for launch accounting; 0 for arguments the call would reject).
 * kv_indices_len is the call's kv_indices_len: the warp-shuffle kernel
 * needs no merge launch when no request can hold more keys than one of its
 * splits takes.
 */
int mla_tree_verify_launch_count(int batch, int total_q, int heads, int64_t kv_indices_len,
                                 int max_splits, int path);

/*
 * Test facility for the kernels' failure detection (the paper has no
 * counterpart; its validate gate is the nearest idea: "Deploying a Custom
 * sm_120 Verify Kernel into Production", "The Validate Mode"). Every wait
 * inside the tensor-core verify kernel is bounded; when one gives up, the
 * kernel sets MT_DEV_TIMEOUT in dev_status, issues no further copy or MMA,
 * drains what is in flight and exits, leaving the device usable.
 *   wait_limit_ns: bound of every such wait, 0 = the default of 2 s.
 *   drop_item:     -1 = off; else the kernel's copy engines issue nothing
 *                  from its work item drop_item on (items number the
 *                  (128-row tile, key split) pairs of a call from 0), so
 *                  the waits on those keys run out.
 * Process-wide: applies to every tensor-core verify call enqueued after it
 * until it is called again with (-1, 0). Returns MT_EINVAL for
 * drop_item < -1 or a negative limit. Not for production use.
 */
int mla_tree_test_wait_limits(int drop_item, int64_t wait_limit_ns);

/*
 * Tree-verify attention ("Flipping the Switch", "The Long Road to Parity"
 * and "The Broader Context"; "Pivot to Live Cutover", "The Technical
 * Investigation" and "Input Knowledge Required"). For every request b, draft
 * row i < n_b (token t = qo_indptr[b] + i) and head h < heads:
 *     s_j  = sm_scale * <q[t, h, 0:576], kv_buf[kv_indices[kv_indptr[b] + j], 0:576]>
 *     vis_j = packed_mask[mask_indptr[b] + i * L_b + j] != 0,    j < L_b
 *     lse[t, h] = ln sum_{vis} exp(s_j)
 *     out[t, h, :] = bf16_rne( sum_{vis} exp(s_j - lse[t, h]) * kv_buf[slot_j, 0:512] )
 * A row with no visible position gets out = 0 and lse = -inf.
 * Arithmetic: every score is an fp32 sum of bf16 products (the tensor-core
 * kernel adds its two CTAs' fp32 partial sums); the online softmax runs in
 * fp32 in the log2 domain; the tensor-core kernel rounds the weights to bf16
 * for its P.V product and sums those same bf16 weights in the denominator,
 * the warp-shuffle kernel keeps them in fp32; split partials are fp32.
 * Nothing narrower than fp32 holds a score or a partial output.
 *   q:       bf16 [total_q, heads, 576], 16-byte aligned
 *   kv_buf:  bf16 [num_slots, 576], 16-byte aligned (rows of 1152 bytes)
 *   kv_indices: int32 [kv_indices_len]; kv_indptr, qo_indptr: int32 [batch+1]
 *   packed_mask: uint8 [mask_len]; mask_indptr: int64 [batch+1]
 *   out:     bf16 [total_q, heads, 512], 16-byte aligned
 *   lse:     fp32 [total_q, heads]
 *   workspace: >= mla_tree_verify_workspace_bytes(batch, total_q, heads,
 *            max_splits) bytes, 256-byte aligned.
 *   max_splits: upper bound on KV splits per request (0 = automatic);
 *            the kernels choose each request's split count on the device.
 *            Results agree across split counts up to fp32 rounding.
 *   path:    0 = automatic, 1 = SIMT (warp-shuffle) kernel, 2 = tensor-core
 *            (tcgen05/TMEM) kernel.
 * Inconsistent device-side sizes set MT_DEV_BAD_INDPTR, out-of-range slots
 * MT_DEV_BAD_SLOT; rows of an inconsistent request are left unwritten.
 */
int mla_tree_verify(const mt_bf16* q, const mt_bf16* kv_buf, int64_t num_slots,
                    const int32_t* kv_indices, int64_t kv_indices_len,
                    const int32_t* kv_indptr, const int32_t* qo_indptr,
                    const uint8_t* packed_mask, int64_t mask_len, const int64_t* mask_indptr,
                    int batch, int total_q, int heads, float sm_scale,
                    mt_bf16* out, float* lse,
                    void* workspace, size_t workspace_bytes, int max_splits, int path,
                    int32_t* dev_status, mt_stream_t stream);

/*
 * mla_tree_verify with the tree mask in the bit form of tree_mask_pack_bits:
 *     vis_j = (mask_words[mask_word_indptr[b] + i * W_b + j / 32] >> (j % 32)) & 1
 * with W_b = ceil(L_b / 32); mask_len_words counts the words of mask_words.
 * Everything else (arguments, outputs, workspace, paths, error behaviour)
 * is that of mla_tree_verify, and the results are the same as for the
 * equivalent byte mask.
 */
int mla_tree_verify_bits(const mt_bf16* q, const mt_bf16* kv_buf, int64_t num_slots,
                         const int32_t* kv_indices, int64_t kv_indices_len,
                         const int32_t* kv_indptr, const int32_t* qo_indptr,
                         const uint32_t* mask_words, int64_t mask_len_words,
                         const int64_t* mask_word_indptr,
                         int batch, int total_q, int heads, float sm_scale,
                         mt_bf16* out, float* lse,
                         void* workspace, size_t workspace_bytes, int max_splits, int path,
                         int32_t* dev_status, mt_stream_t stream);

/*
 * Mask options of mla_tree_verify_masked ("The Pivot to Live Cutover",
 * section "The Technical Investigation: Probing the Integration Surface":
 * the serving engine's attention kernel takes the tree mask with a switch
 * that leaves the mask unread over the prefix columns).
 *   MT_MASK_BITS         the mask is in the bit form of tree_mask_pack_bits
 *                        (uint32 words; mask_len counts words), else bytes
 *   MT_MASK_SKIP_PREFIX  columns j < P_b = L_b - n_b (the prefix) are
 *                        visible to every draft row; their mask entries are
 *                        never read and may hold anything. The layout of the
 *                        mask (row stride L_b bytes or ceil(L_b / 32) words)
 *                        is unchanged.
 */
#define MT_MASK_BITS 1
#define MT_MASK_SKIP_PREFIX 2

/*
 * mla_tree_verify with the mask form and options as flags (a combination of
 * MT_MASK_BITS and MT_MASK_SKIP_PREFIX; other bits give MT_EINVAL):
 *     vis_j = 1                                   if SKIP_PREFIX and j < P_b
 *           = the mask entry (i, j) of that form   otherwise
 * mask: uint8 [mask_len] bytes, or uint32 [mask_len] words (4-byte aligned)
 * with MT_MASK_BITS. flags 0 is mla_tree_verify, MT_MASK_BITS is
 * mla_tree_verify_bits; everything else (arguments, outputs, workspace,
 * paths, error behaviour) is theirs.
 */
int mla_tree_verify_masked(const mt_bf16* q, const mt_bf16* kv_buf, int64_t num_slots,
                           const int32_t* kv_indices, int64_t kv_indices_len,
                           const int32_t* kv_indptr, const int32_t* qo_indptr,
                           const void* mask, int64_t mask_len, const int64_t* mask_indptr,
                           int mask_flags, int batch, int total_q, int heads, float sm_scale,
                           mt_bf16* out, float* lse,
                           void* workspace, size_t workspace_bytes, int max_splits, int path,
                           int32_t* dev_status, mt_stream_t stream);

/*
 * Validate mode ("Deploying a Custom sm_120 Verify Kernel into Production",
 * "The Validate Mode": the custom kernel runs next to the reference path on
 * the same tensors and the difference is reported). A debug entry point:
 * the same call as mla_tree_verify, computed twice, by the tensor-core
 * kernel into out / lse (what the caller gets) and by the warp-shuffle
 * kernel into scratch inside the workspace; then, on the device,
 *   diff[0] = max over elements |out_tc - out_simt|            (fp32 of bf16)
 *   diff[1] = max over rows |lse_tc - lse_simt| / max(1, |lse_tc|)
 *            (rows where both are -inf count 0; one -inf counts +inf)
 * and MT_DEV_MISMATCH is set in dev_status when either exceeds tolerance.
 *   diff: fp32 [2] device memory, overwritten by the call.
 *   workspace: >= mla_tree_verify_validate_workspace_bytes(batch, total_q,
 *            heads, max_splits) bytes, 256-byte aligned.
 * Returns MT_EUNSUPPORTED when the tensor-core kernel cannot serve the call.
 * The gate in "Deploying a Custom sm_120 Verify Kernel into Production"
 * compared against the serving engine's own attention backend; here the two
 * paths are this library's own, written independently.
 */
size_t mla_tree_verify_validate_workspace_bytes(int batch, int total_q, int heads, int max_splits);
int mla_tree_verify_validate(const mt_bf16* q, const mt_bf16* kv_buf, int64_t num_slots,
                             const int32_t* kv_indices, int64_t kv_indices_len,
                             const int32_t* kv_indptr, const int32_t* qo_indptr,
                             const uint8_t* packed_mask, int64_t mask_len,
                             const int64_t* mask_indptr, int batch, int total_q, int heads,
                             float sm_scale, mt_bf16* out, float* lse, void* workspace,
                             size_t workspace_bytes, int max_splits, float tolerance,
                             float* diff, int32_t* dev_status, mt_stream_t stream);

/*
 * mla_tree_verify without a caller-provided workspace. The paper has no
 * counterpart: this exists for embedders. Some callers cannot allocate
 * device memory at all: an engine that reserves the whole GPU up front and
 * hands out memory only from its own arena, a plugin living in a process
 * whose allocator it does not own, or a latency-critical path that cannot
 * afford cudaMalloc's implicit synchronisation. This entry point computes
 * exactly what mla_tree_verify computes, with the same arguments minus
 * workspace/workspace_bytes; its scratch lives in a fixed array of
 * MT_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU that
 * loads the library keeps until the process exits. It never allocates.
 *   - A request whose scratch (mla_tree_verify_workspace_bytes for the same
 *     batch, total_q, heads, max_splits) exceeds MT_NOALLOC_SCRATCH_BYTES is
 *     rejected with MT_ESCRATCH before anything is launched.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address with a runtime query.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents (nothing in it needs clearing). Calls that may overlap on the
 *     GPU -- unordered streams -- race on it; order them.
 *   - The looked-up address is kept for the life of the process: after
 *     cudaDeviceReset on a device, the library must not be used on that
 *     device again (its cached per-device state, this address included,
 *     would be stale).
 */
#define MT_NOALLOC_SCRATCH_BYTES (64u << 20)
int mla_tree_verify_noalloc(const mt_bf16* q, const mt_bf16* kv_buf, int64_t num_slots,
                            const int32_t* kv_indices, int64_t kv_indices_len,
                            const int32_t* kv_indptr, const int32_t* qo_indptr,
                            const uint8_t* packed_mask, int64_t mask_len, const int64_t* mask_indptr,
                            int batch, int total_q, int heads, float sm_scale,
                            mt_bf16* out, float* lse, int max_splits, int path,
                            int32_t* dev_status, mt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_TREE_H */
