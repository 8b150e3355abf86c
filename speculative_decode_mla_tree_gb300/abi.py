"""ctypes binding of libmla_tree.so: same names as the C ABI, argument
marshalling only (torch tensors -> device pointers, the current stream).
Every step of the verify path runs in the library's kernels; when the
library is missing this module raises instead of computing anything."""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libmla_tree.so")

MT_OK, MT_EINVAL, MT_EUNSUPPORTED, MT_EWORKSPACE, MT_ECUDA = 0, -1, -2, -3, -4
DEV_BAD_SLOT, DEV_BAD_PARENT, DEV_BAD_INDPTR, DEV_TREE_TOO_BIG, DEV_TIMEOUT = 1, 2, 4, 8, 16
DEV_MISMATCH = 32
PATH_AUTO, PATH_SIMT, PATH_TC = 0, 1, 2

EXPORTS = ["mla_tree_abi_version", "mla_tree_status_string", "mla_tree_draft_kv_scatter",
           "mla_tree_kv_indices_build", "tree_mask_pack", "tree_mask_pack_bits", "mla_tree_prepare",
           "mla_tree_verify_workspace_bytes", "mla_tree_verify_launch_count", "mla_tree_verify",
           "mla_tree_verify_bits", "mla_tree_verify_masked", "mla_tree_verify_validate_workspace_bytes",
           "mla_tree_verify_validate", "mla_tree_verify_noalloc", "mla_tree_test_wait_limits"]
MT_ESCRATCH = -5
NOALLOC_SCRATCH_BYTES = 64 << 20

_lib = None
P = ctypes.c_void_p
I32, I64, SZ, F32 = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float


class MlaTreeError(RuntimeError):
    pass


def load():
    """Load the library once; fail loudly if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise MlaTreeError("libmla_tree.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    lib.mla_tree_abi_version.restype = I32
    lib.mla_tree_status_string.restype = ctypes.c_char_p
    lib.mla_tree_status_string.argtypes = [I32]
    lib.mla_tree_draft_kv_scatter.restype = I32
    lib.mla_tree_draft_kv_scatter.argtypes = [P, I64, P, I32, P, I64, P, P]
    lib.mla_tree_kv_indices_build.restype = I32
    lib.mla_tree_kv_indices_build.argtypes = [P, I64, P, P, P, I32, I32, P, I64, P, P, P]
    lib.tree_mask_pack.restype = I32
    lib.tree_mask_pack.argtypes = [P, P, P, I32, I32, P, P, I64, P, P]
    lib.tree_mask_pack_bits.restype = I32
    lib.tree_mask_pack_bits.argtypes = [P, P, P, I32, I32, P, P, I64, P, P]
    lib.mla_tree_prepare.restype = I32
    lib.mla_tree_prepare.argtypes = [P, I64, P, P, I64, P, P, P, I32, I32, P, I64, P, I64, P, P, P, I64,
                                     P, P]
    lib.mla_tree_verify_workspace_bytes.restype = SZ
    lib.mla_tree_verify_workspace_bytes.argtypes = [I32, I32, I32, I32]
    lib.mla_tree_verify_launch_count.restype = I32
    lib.mla_tree_verify_launch_count.argtypes = [I32, I32, I32, I64, I32, I32]
    lib.mla_tree_verify.restype = I32
    lib.mla_tree_verify.argtypes = [P, P, I64, P, I64, P, P, P, I64, P, I32, I32, I32, F32,
                                    P, P, P, SZ, I32, I32, P, P]
    lib.mla_tree_verify_bits.restype = I32
    lib.mla_tree_verify_bits.argtypes = [P, P, I64, P, I64, P, P, P, I64, P, I32, I32, I32, F32,
                                         P, P, P, SZ, I32, I32, P, P]
    lib.mla_tree_verify_masked.restype = I32
    lib.mla_tree_verify_masked.argtypes = [P, P, I64, P, I64, P, P, P, I64, P, I32, I32, I32, I32, F32,
                                           P, P, P, SZ, I32, I32, P, P]
    lib.mla_tree_verify_validate_workspace_bytes.restype = SZ
    lib.mla_tree_verify_validate_workspace_bytes.argtypes = [I32, I32, I32, I32]
    lib.mla_tree_verify_validate.restype = I32
    lib.mla_tree_verify_validate.argtypes = [P, P, I64, P, I64, P, P, P, I64, P, I32, I32, I32, F32,
                                             P, P, P, SZ, I32, F32, P, P, P]
    lib.mla_tree_test_wait_limits.restype = I32
    lib.mla_tree_test_wait_limits.argtypes = [I32, I64]
    lib.mla_tree_verify_noalloc.restype = I32
    lib.mla_tree_verify_noalloc.argtypes = [P, P, I64, P, I64, P, P, P, I64, P, I32, I32, I32, F32,
                                            P, P, I32, I32, P, P]
    _lib = lib
    return lib


def _check(rc, what):
    if rc != MT_OK:
        msg = load().mla_tree_status_string(rc).decode()
        raise MlaTreeError("%s failed: %d (%s)" % (what, rc, msg))


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise MlaTreeError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise MlaTreeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise MlaTreeError("%s must be contiguous" % name)
    return t.data_ptr() if t.numel() else None


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def abi_version():
    return load().mla_tree_abi_version()


def mla_tree_draft_kv_scatter(src, out_cache_loc, kv_buf, status=None, stream=None):
    """kv_buf[out_cache_loc[t]] = src[t] for every draft token t."""
    if src.dim() != 2 or src.stride(1) != 1 or src.dtype != torch.bfloat16 or not src.is_cuda:
        raise MlaTreeError("src must be a CUDA bf16 [T, >=576] tensor with unit column stride")
    rc = load().mla_tree_draft_kv_scatter(src.data_ptr() if src.numel() else None, src.stride(0),
                                          _ptr(out_cache_loc, torch.int32, "out_cache_loc"),
                                          out_cache_loc.numel(), _ptr(kv_buf, torch.bfloat16, "kv_buf"),
                                          kv_buf.shape[0], _ptr(status, torch.int32, "status"),
                                          _stream(stream))
    _check(rc, "mla_tree_draft_kv_scatter")


def mla_tree_kv_indices_build(prefix_indices, prefix_indptr, out_cache_loc, qo_indptr,
                              kv_indices, kv_indptr, status=None, stream=None):
    """kv_indices = per request, prefix slots followed by draft slots."""
    batch = qo_indptr.numel() - 1
    rc = load().mla_tree_kv_indices_build(
        _ptr(prefix_indices, torch.int32, "prefix_indices"), prefix_indices.numel(),
        _ptr(prefix_indptr, torch.int32, "prefix_indptr"),
        _ptr(out_cache_loc, torch.int32, "out_cache_loc"), _ptr(qo_indptr, torch.int32, "qo_indptr"),
        batch, out_cache_loc.numel(), _ptr(kv_indices, torch.int32, "kv_indices"), kv_indices.numel(),
        _ptr(kv_indptr, torch.int32, "kv_indptr"), _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "mla_tree_kv_indices_build")


def tree_mask_pack(parents, qo_indptr, kv_indptr, mask_indptr, packed_mask, status=None, stream=None):
    """Ancestor-or-self tree mask, row stride prefix + draft, flat per request."""
    batch = qo_indptr.numel() - 1
    rc = load().tree_mask_pack(
        _ptr(parents, torch.int32, "parents"), _ptr(qo_indptr, torch.int32, "qo_indptr"),
        _ptr(kv_indptr, torch.int32, "kv_indptr"), batch, parents.numel(),
        _ptr(mask_indptr, torch.int64, "mask_indptr"), _ptr(packed_mask, torch.uint8, "packed_mask"),
        packed_mask.numel(), _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "tree_mask_pack")


def tree_mask_pack_bits(parents, qo_indptr, kv_indptr, mask_word_indptr, mask_words, status=None,
                        stream=None):
    """The same tree mask, one bit per (row, column): rows of ceil(L/32) uint32 words."""
    batch = qo_indptr.numel() - 1
    rc = load().tree_mask_pack_bits(
        _ptr(parents, torch.int32, "parents"), _ptr(qo_indptr, torch.int32, "qo_indptr"),
        _ptr(kv_indptr, torch.int32, "kv_indptr"), batch, parents.numel(),
        _ptr(mask_word_indptr, torch.int64, "mask_word_indptr"),
        _ptr(mask_words, torch.int32, "mask_words"), mask_words.numel(),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "tree_mask_pack_bits")


def mla_tree_prepare(draft_kv, out_cache_loc, prefix_indices, prefix_indptr, qo_indptr, parents,
                     kv_buf, kv_indices, kv_indptr, mask_word_indptr, mask_words, status=None,
                     stream=None):
    """Draft-KV scatter, KV index marshaling and bit-form mask packing in one launch."""
    if (draft_kv.dim() != 2 or draft_kv.stride(1) != 1 or draft_kv.dtype != torch.bfloat16
            or not draft_kv.is_cuda):
        raise MlaTreeError("draft_kv must be a CUDA bf16 [T, >=576] tensor with unit column stride")
    batch = qo_indptr.numel() - 1
    rc = load().mla_tree_prepare(
        draft_kv.data_ptr() if draft_kv.numel() else None, draft_kv.stride(0),
        _ptr(out_cache_loc, torch.int32, "out_cache_loc"),
        _ptr(prefix_indices, torch.int32, "prefix_indices"), prefix_indices.numel(),
        _ptr(prefix_indptr, torch.int32, "prefix_indptr"), _ptr(qo_indptr, torch.int32, "qo_indptr"),
        _ptr(parents, torch.int32, "parents"), batch, out_cache_loc.numel(),
        _ptr(kv_buf, torch.bfloat16, "kv_buf"), kv_buf.shape[0],
        _ptr(kv_indices, torch.int32, "kv_indices"), kv_indices.numel(),
        _ptr(kv_indptr, torch.int32, "kv_indptr"),
        _ptr(mask_word_indptr, torch.int64, "mask_word_indptr"),
        _ptr(mask_words, torch.int32, "mask_words"), mask_words.numel(),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "mla_tree_prepare")


def mla_tree_test_wait_limits(drop_item=-1, wait_limit_ns=0):
    """Test facility: bound every wait of the tensor-core kernel by
    wait_limit_ns (0 = the default) and make its copy engines issue nothing
    from work item drop_item on (-1 = off). Process-wide."""
    _check(load().mla_tree_test_wait_limits(int(drop_item), int(wait_limit_ns)),
           "mla_tree_test_wait_limits")


def mla_tree_verify_workspace_bytes(batch, total_q, heads, max_splits=0):
    return int(load().mla_tree_verify_workspace_bytes(batch, total_q, heads, max_splits))


def mla_tree_verify_launch_count(batch, total_q, heads, kv_indices_len, max_splits=0, path=PATH_AUTO):
    return int(load().mla_tree_verify_launch_count(batch, total_q, heads, kv_indices_len, max_splits, path))


def mla_tree_verify(q, kv_buf, kv_indices, kv_indptr, qo_indptr, packed_mask, mask_indptr,
                    sm_scale, out, lse, workspace, max_splits=0, path=PATH_AUTO, status=None,
                    stream=None):
    """Tree-verify attention: out [T, H, 512] bf16 and lse [T, H] fp32."""
    if q.dim() != 3 or q.shape[2] != 576:
        raise MlaTreeError("q must be [total_q, heads, 576]")
    total_q, heads = q.shape[0], q.shape[1]
    batch = qo_indptr.numel() - 1
    rc = load().mla_tree_verify(
        _ptr(q, torch.bfloat16, "q"), _ptr(kv_buf, torch.bfloat16, "kv_buf"), kv_buf.shape[0],
        _ptr(kv_indices, torch.int32, "kv_indices"), kv_indices.numel(),
        _ptr(kv_indptr, torch.int32, "kv_indptr"), _ptr(qo_indptr, torch.int32, "qo_indptr"),
        _ptr(packed_mask, torch.uint8, "packed_mask"), packed_mask.numel(),
        _ptr(mask_indptr, torch.int64, "mask_indptr"), batch, total_q, heads, float(sm_scale),
        _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), max_splits, path,
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "mla_tree_verify")


def mla_tree_verify_bits(q, kv_buf, kv_indices, kv_indptr, qo_indptr, mask_words, mask_word_indptr,
                         sm_scale, out, lse, workspace, max_splits=0, path=PATH_AUTO, status=None,
                         stream=None):
    """mla_tree_verify with the mask in the bit form of tree_mask_pack_bits
    (mask_words: int32 tensor holding the uint32 words)."""
    if q.dim() != 3 or q.shape[2] != 576:
        raise MlaTreeError("q must be [total_q, heads, 576]")
    total_q, heads = q.shape[0], q.shape[1]
    batch = qo_indptr.numel() - 1
    rc = load().mla_tree_verify_bits(
        _ptr(q, torch.bfloat16, "q"), _ptr(kv_buf, torch.bfloat16, "kv_buf"), kv_buf.shape[0],
        _ptr(kv_indices, torch.int32, "kv_indices"), kv_indices.numel(),
        _ptr(kv_indptr, torch.int32, "kv_indptr"), _ptr(qo_indptr, torch.int32, "qo_indptr"),
        _ptr(mask_words, torch.int32, "mask_words"), mask_words.numel(),
        _ptr(mask_word_indptr, torch.int64, "mask_word_indptr"), batch, total_q, heads,
        float(sm_scale), _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), max_splits, path,
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "mla_tree_verify_bits")


MASK_BITS = 1         # the mask is in the bit form (int32 tensor of uint32 words)
MASK_SKIP_PREFIX = 2  # prefix columns visible, their mask entries unread


def mla_tree_verify_masked(q, kv_buf, kv_indices, kv_indptr, qo_indptr, mask, mask_indptr,
                           mask_flags, sm_scale, out, lse, workspace, max_splits=0, path=PATH_AUTO,
                           status=None, stream=None):
    """mla_tree_verify with the mask form and options as flags (MASK_BITS,
    MASK_SKIP_PREFIX): mask is a uint8 byte mask, or int32 words with
    MASK_BITS."""
    if q.dim() != 3 or q.shape[2] != 576:
        raise MlaTreeError("q must be [total_q, heads, 576]")
    total_q, heads = q.shape[0], q.shape[1]
    batch = qo_indptr.numel() - 1
    mdt = torch.int32 if mask_flags & MASK_BITS else torch.uint8
    rc = load().mla_tree_verify_masked(
        _ptr(q, torch.bfloat16, "q"), _ptr(kv_buf, torch.bfloat16, "kv_buf"), kv_buf.shape[0],
        _ptr(kv_indices, torch.int32, "kv_indices"), kv_indices.numel(),
        _ptr(kv_indptr, torch.int32, "kv_indptr"), _ptr(qo_indptr, torch.int32, "qo_indptr"),
        _ptr(mask, mdt, "mask"), mask.numel(), _ptr(mask_indptr, torch.int64, "mask_indptr"),
        int(mask_flags), batch, total_q, heads, float(sm_scale), _ptr(out, torch.bfloat16, "out"),
        _ptr(lse, torch.float32, "lse"), _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        max_splits, path, _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "mla_tree_verify_masked")


def mla_tree_verify_validate_workspace_bytes(batch, total_q, heads, max_splits=0):
    return int(load().mla_tree_verify_validate_workspace_bytes(batch, total_q, heads, max_splits))


def mla_tree_verify_validate(q, kv_buf, kv_indices, kv_indptr, qo_indptr, packed_mask, mask_indptr,
                             sm_scale, out, lse, workspace, diff, tolerance=1e-2, max_splits=0,
                             status=None, stream=None):
    """Validate mode: the call computed by both kernels; out/lse get the
    tensor-core result, diff (fp32 [2] on the device) the max-abs output and
    max relative LSE differences, status MT_DEV_MISMATCH beyond tolerance."""
    if q.dim() != 3 or q.shape[2] != 576:
        raise MlaTreeError("q must be [total_q, heads, 576]")
    total_q, heads = q.shape[0], q.shape[1]
    batch = qo_indptr.numel() - 1
    rc = load().mla_tree_verify_validate(
        _ptr(q, torch.bfloat16, "q"), _ptr(kv_buf, torch.bfloat16, "kv_buf"), kv_buf.shape[0],
        _ptr(kv_indices, torch.int32, "kv_indices"), kv_indices.numel(),
        _ptr(kv_indptr, torch.int32, "kv_indptr"), _ptr(qo_indptr, torch.int32, "qo_indptr"),
        _ptr(packed_mask, torch.uint8, "packed_mask"), packed_mask.numel(),
        _ptr(mask_indptr, torch.int64, "mask_indptr"), batch, total_q, heads, float(sm_scale),
        _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), max_splits, float(tolerance),
        _ptr(diff, torch.float32, "diff"), _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "mla_tree_verify_validate")


def mla_tree_verify_noalloc(q, kv_buf, kv_indices, kv_indptr, qo_indptr, packed_mask, mask_indptr,
                            sm_scale, out, lse, max_splits=0, path=PATH_AUTO, status=None,
                            stream=None):
    """mla_tree_verify for callers that cannot allocate: the split scratch is
    the library's built-in static device buffer instead of a workspace."""
    if q.dim() != 3 or q.shape[2] != 576:
        raise MlaTreeError("q must be [total_q, heads, 576]")
    total_q, heads = q.shape[0], q.shape[1]
    batch = qo_indptr.numel() - 1
    rc = load().mla_tree_verify_noalloc(
        _ptr(q, torch.bfloat16, "q"), _ptr(kv_buf, torch.bfloat16, "kv_buf"), kv_buf.shape[0],
        _ptr(kv_indices, torch.int32, "kv_indices"), kv_indices.numel(),
        _ptr(kv_indptr, torch.int32, "kv_indptr"), _ptr(qo_indptr, torch.int32, "qo_indptr"),
        _ptr(packed_mask, torch.uint8, "packed_mask"), packed_mask.numel(),
        _ptr(mask_indptr, torch.int64, "mask_indptr"), batch, total_q, heads, float(sm_scale),
        _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"), max_splits, path,
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "mla_tree_verify_noalloc")
