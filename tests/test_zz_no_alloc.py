"""mla_tree_verify_noalloc, the entry point for callers that cannot allocate
device memory (engines that own every byte of the GPU, plugins inside a host
whose allocator they do not control, paths that cannot afford cudaMalloc's
synchronisation). It must give what the regular entry point gives on the
same inputs, on two calls in a row (the shared static scratch keeps the
previous call's contents), and reject requests larger than its buffer.

This file is collected last on purpose."""
import ctypes

import pytest
import torch

import __graft_entry__
from speculative_decode_mla_tree_gb300 import abi, workloads as W
from speculative_decode_mla_tree_gb300.step import VerifyStep

from parity import LSE_REL, OUT_MAX_ABS, OUT_MEAN_ABS

pytestmark = pytest.mark.gpu


def _noalloc_raw(st, out, lse, max_splits, path):
    """Call the C entry point directly through ctypes (no binding helper)."""
    lib = abi.load()
    return lib.mla_tree_verify_noalloc(
        st.q.data_ptr(), st.pool.data_ptr(), st.pool.shape[0], st.kv_indices.data_ptr(),
        st.kv_indices.numel(), st.kv_indptr.data_ptr(), st.qo_indptr.data_ptr(),
        st.mask.data_ptr(), st.mask.numel(), st.mask_indptr.data_ptr(), st.w.batch, st.w.total_q,
        st.heads, ctypes.c_float(st.sm_scale), out.data_ptr(), lse.data_ptr(), max_splits, path,
        st.status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _agree(out_a, lse_a, out_b, lse_b):
    d = (out_a.float() - out_b.float()).abs()
    assert float(d.max()) <= OUT_MAX_ABS and float(d.mean()) <= OUT_MEAN_ABS
    fin = torch.isfinite(lse_b)
    assert torch.equal(fin, torch.isfinite(lse_a))
    rel = (lse_a[fin] - lse_b[fin]).abs() / lse_b[fin].abs().clamp(min=1.0)
    assert rel.numel() == 0 or float(rel.max()) <= LSE_REL


PATHS = [pytest.param(abi.PATH_SIMT, id="simt"), pytest.param(abi.PATH_TC, id="tcgen05"),
         pytest.param(abi.PATH_AUTO, id="auto")]


@pytest.mark.parametrize("path", PATHS)
def test_noalloc_matches_workspace_entry_point_twice(path):
    """Two calls in a row: the first splits 1152 (node, head) rows over up to
    16 splits per request, the second covers fewer tokens and splits, so it
    runs on scratch that still holds the first call's partials and counts."""
    __graft_entry__.build()
    cases = [(W.make_workload("na1", 16, [3000, 1200, 500], "uniform", [32, 16, 24], 16384, seed=42), 16),
             (W.make_workload("na2", 8, [900, 300], "uniform", [16, 16], 8192, seed=43), 4)]
    for w, splits in cases:
        st = VerifyStep(w, max_splits=splits, path=path)
        st.run()                       # regular entry point with a caller workspace
        out = torch.empty_like(st.out)
        lse = torch.empty_like(st.lse)
        rc = _noalloc_raw(st, out, lse, splits, path)
        assert rc == abi.MT_OK, rc
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        _agree(out, lse, st.out, st.lse)


@pytest.mark.parametrize("splits", [1, 0], ids=["unsplit", "auto"])
def test_noalloc_serves_unsplit_large_batches(splits):
    """32 requests x 64 nodes x 64 heads (131072 rows): unsplit, and with the
    automatic split choice (which is one split here), the call needs only
    the per-token split counts and fits the built-in scratch."""
    __graft_entry__.build()
    w = W.config(3)
    need = abi.mla_tree_verify_workspace_bytes(w.batch, w.total_q, w.heads, splits)
    assert need <= abi.NOALLOC_SCRATCH_BYTES
    st = VerifyStep(w, max_splits=splits, path=abi.PATH_TC)
    st.run()
    out = torch.empty_like(st.out)
    lse = torch.empty_like(st.lse)
    assert _noalloc_raw(st, out, lse, splits, abi.PATH_TC) == abi.MT_OK
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    _agree(out, lse, st.out, st.lse)


def test_noalloc_rejects_requests_beyond_its_buffer():
    __graft_entry__.build()
    w = W.make_workload("big", 64, [64], "uniform", [64], 4096, seed=43)
    st = VerifyStep(w, max_splits=1, path=abi.PATH_SIMT)
    need = abi.mla_tree_verify_workspace_bytes(w.batch, w.total_q, w.heads, 64)
    assert need > abi.NOALLOC_SCRATCH_BYTES
    out = torch.empty_like(st.out)
    lse = torch.empty_like(st.lse)
    assert _noalloc_raw(st, out, lse, 64, abi.PATH_SIMT) == abi.MT_ESCRATCH
