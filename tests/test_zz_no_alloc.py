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


def test_noalloc_matches_workspace_entry_point_twice():
    __graft_entry__.build()
    cases = [(W.small(seed=41), 8),
             (W.make_workload("na", 8, [900, 2500], "uniform", [16, 12], 8192, seed=42), 16)]
    for w, splits in cases:            # two calls in a row, different shapes
        st = VerifyStep(w, max_splits=splits, path=abi.PATH_SIMT)
        st.run()                       # regular entry point with a caller workspace
        out = torch.empty_like(st.out)
        lse = torch.empty_like(st.lse)
        rc = _noalloc_raw(st, out, lse, splits, abi.PATH_SIMT)
        assert rc == abi.MT_OK, rc
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
